// prox_prepare.cu -- one-off per-layer preparation (not on the timed path).
//
// "Prox" (Abstract): Stage 1 reads quantized proxy copies of W_gate and W_up;
// Stage 2 reads the selected gate/up rows and down-projection columns.  This
// file builds:
//   * the int4 group-128 symmetric proxy, packed input-dim-major so that one
//     kept input dimension is one contiguous row of d_ff bytes;
//   * the channel-interleaved gate|up rows and the channel-major W_down^T,
//     either as bf16 copies or quantized per row to int8 or int4 (symmetric,
//     one fp32 scale amax / 127 or amax / 7 per row; the scales travel at the
//     end of each gate|up row so that one bulk copy brings a channel's codes
//     and scales).
#include "prox_internal.cuh"

namespace prox {
namespace {

// One thread per (channel c, group g): fp16 scales for gate and up, then the
// 128 code bytes of the group, written as column c of rows [128g, 128g+128).
__global__ void __launch_bounds__(128)
k_quantize_pack(const __nv_bfloat16* __restrict__ w_gate, const __nv_bfloat16* __restrict__ w_up,
                uint8_t* __restrict__ codes, __half2* __restrict__ scales, int d, int F, int Fp) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    const int g = blockIdx.y;
    if (c >= Fp) return;
    uint8_t* col = codes + (size_t)(g * kGroup) * Fp + c;
    if (c >= F) {  // padding channel: code 0 for both nibbles, scale 0
        for (int t = 0; t < kGroup; ++t) col[(size_t)t * Fp] = 0x88;
        scales[(size_t)g * Fp + c] = __floats2half2_rn(0.0f, 0.0f);
        return;
    }
    const __nv_bfloat16* rg = w_gate + (size_t)c * d + g * kGroup;
    const __nv_bfloat16* ru = w_up + (size_t)c * d + g * kGroup;
    float amax_g = 0.0f, amax_u = 0.0f;
    for (int t = 0; t < kGroup; ++t) {
        amax_g = fmaxf(amax_g, fabsf(__bfloat162float(rg[t])));
        amax_u = fmaxf(amax_u, fabsf(__bfloat162float(ru[t])));
    }
    // s = fp16_rne(fl32(amax / 7)); correctly rounded binary32 division
    const __half sg = __float2half_rn(__fdiv_rn(amax_g, 7.0f));
    const __half su = __float2half_rn(__fdiv_rn(amax_u, 7.0f));
    scales[(size_t)g * Fp + c] = __halves2half2(sg, su);
    const float sgf = __half2float(sg), suf = __half2float(su);
    for (int t = 0; t < kGroup; ++t) {
        int qg = 0, qu = 0;
        if (sgf != 0.0f) qg = min(7, max(-8, __float2int_rn(__fdiv_rn(__bfloat162float(rg[t]), sgf))));
        if (suf != 0.0f) qu = min(7, max(-8, __float2int_rn(__fdiv_rn(__bfloat162float(ru[t]), suf))));
        col[(size_t)t * Fp] = (uint8_t)((qg + 8) | ((qu + 8) << 4));
    }
}

// W_down [d][F] -> down_t [F][d], 32x32 tiles through shared memory.
__global__ void __launch_bounds__(256)
k_transpose(const __nv_bfloat16* __restrict__ src, __nv_bfloat16* __restrict__ dst, int rows,
            int cols) {
    __shared__ __nv_bfloat16 tile[32][33];
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    for (int i = ty; i < 32; i += 8) {
        const int r = r0 + i, c = c0 + tx;
        if (r < rows && c < cols) tile[i][tx] = src[(size_t)r * cols + c];
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int c = c0 + i, r = r0 + tx;
        if (c < cols && r < rows) dst[(size_t)c * rows + r] = tile[tx][i];
    }
}

// Row codes: int8 (WQ = 1) = round-to-nearest-even of the binary32 quotient
// w / s clamped to [-127, 127] with s = amax / 127; int4 (WQ = 2) the same
// with s = amax / 7, clamped to [-8, 7].  0 on an all-zero row.
template <int WQ>
__device__ __forceinline__ int row_code(float w, float s) {
    if (s == 0.0f) return 0;
    const int q = __float2int_rn(__fdiv_rn(w, s));
    return WQ == 2 ? min(7, max(-8, q)) : min(127, max(-127, q));
}
template <int WQ>
__device__ __forceinline__ float row_scale(float amax) {
    return __fdiv_rn(amax, WQ == 2 ? 7.0f : 127.0f);
}

// int4 word of 8 consecutive codes (offset binary n = q + 8): element
// 2 j + h in bits 16 h + 4 j.
__device__ __forceinline__ uint32_t pack_q4(const int* q) {
    uint32_t w = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) w |= (uint32_t)(q[e] + 8) << (16 * (e & 1) + 4 * (e >> 1));
    return w;
}

// One CTA per channel c: the gate and up codes of c and their scales, row c
// of the output = codes of gate | codes of up | s_gate s_up s_down 0
// (int8: 2 d bytes of codes, int4: d bytes; s_down is written by
// k_rowq_down).
template <int WQ>
__global__ void __launch_bounds__(256)
k_rowq_gateup(const __nv_bfloat16* __restrict__ w_gate, const __nv_bfloat16* __restrict__ w_up,
              uint8_t* __restrict__ out, int d) {
    __shared__ float red[2][8];
    const int c = blockIdx.x, tid = threadIdx.x;
    const __nv_bfloat16* rg = w_gate + (size_t)c * d;
    const __nv_bfloat16* ru = w_up + (size_t)c * d;
    float ag = 0.0f, au = 0.0f;
    for (int j = tid; j < d; j += 256) {
        ag = fmaxf(ag, fabsf(__bfloat162float(rg[j])));
        au = fmaxf(au, fabsf(__bfloat162float(ru[j])));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ag = fmaxf(ag, __shfl_xor_sync(0xffffffffu, ag, o));
        au = fmaxf(au, __shfl_xor_sync(0xffffffffu, au, o));
    }
    if ((tid & 31) == 0) {
        red[0][tid >> 5] = ag;
        red[1][tid >> 5] = au;
    }
    __syncthreads();
    float mg = 0.0f, mu = 0.0f;
    for (int w = 0; w < 8; ++w) {
        mg = fmaxf(mg, red[0][w]);
        mu = fmaxf(mu, red[1][w]);
    }
    const float sg = row_scale<WQ>(mg), su = row_scale<WQ>(mu);
    uint8_t* row = out + (size_t)c * gu_row_bytes(d, WQ);
    if constexpr (WQ == 2) {
        uint32_t* qg = reinterpret_cast<uint32_t*>(row);
        uint32_t* qu = qg + d / 8;
        for (int ch = tid; ch < d / 8; ch += 256) {
            int cg[8], cu[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                cg[e] = row_code<WQ>(__bfloat162float(rg[8 * ch + e]), sg);
                cu[e] = row_code<WQ>(__bfloat162float(ru[8 * ch + e]), su);
            }
            qg[ch] = pack_q4(cg);
            qu[ch] = pack_q4(cu);
        }
    } else {
        int8_t* qg = reinterpret_cast<int8_t*>(row);
        int8_t* qu = qg + d;
        for (int j = tid; j < d; j += 256) {
            qg[j] = (int8_t)row_code<WQ>(__bfloat162float(rg[j]), sg);
            qu[j] = (int8_t)row_code<WQ>(__bfloat162float(ru[j]), su);
        }
    }
    if (tid == 0) {
        float* t = reinterpret_cast<float*>(row + gu_row_bytes(d, WQ) - 16);
        t[0] = sg;
        t[1] = su;
        t[3] = 0.0f;
    }
}

// W_down [d][F] -> W_down^T codes [F][down_row_bytes], one scale per channel
// (a column of W_down): 32 channels per CTA, the column maxima first, then
// 32 x 32 tiles through shared memory.  s_down[c] goes to the scale slot of
// gate|up row c.
template <int WQ>
__global__ void __launch_bounds__(256)
k_rowq_down(const __nv_bfloat16* __restrict__ w_down, uint8_t* __restrict__ down_q,
            uint8_t* __restrict__ gateup_q, int d, int F) {
    __shared__ float tile[32][33];
    __shared__ float red[8][32];
    __shared__ float sc[32];
    const int c0 = blockIdx.x * 32, tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int c = c0 + tx;
    float amax = 0.0f;
    if (c < F)
        for (int r = ty; r < d; r += 8)
            amax = fmaxf(amax, fabsf(__bfloat162float(w_down[(size_t)r * F + c])));
    red[ty][tx] = amax;
    __syncthreads();
    if (ty == 0) {
        float m = red[0][tx];
        for (int j = 1; j < 8; ++j) m = fmaxf(m, red[j][tx]);
        const float sd = row_scale<WQ>(m);
        sc[tx] = sd;
        if (c < F)
            *reinterpret_cast<float*>(gateup_q + (size_t)c * gu_row_bytes(d, WQ) +
                                      gu_row_bytes(d, WQ) - 8) = sd;
    }
    __syncthreads();
    for (int r0 = 0; r0 < d; r0 += 32) {  // d is a multiple of 128
        for (int i = ty; i < 32; i += 8)
            tile[i][tx] = c < F ? __bfloat162float(w_down[(size_t)(r0 + i) * F + c]) : 0.0f;
        __syncthreads();
        if constexpr (WQ == 2) {
            // 32 channels x 4 words of 8 codes: thread t < 128 packs word
            // t & 3 of channel c0 + (t >> 2)
            const int t = threadIdx.x, i = t >> 2, wd = t & 3, cc = c0 + i;
            if (t < 128 && cc < F) {
                int q[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) q[e] = row_code<WQ>(tile[8 * wd + e][i], sc[i]);
                reinterpret_cast<uint32_t*>(down_q + (size_t)cc * (d / 2))[(r0 / 8) + wd] = pack_q4(q);
            }
        } else {
            for (int i = ty; i < 32; i += 8) {
                const int cc = c0 + i;
                if (cc < F) down_q[(size_t)cc * d + r0 + tx] = (uint8_t)row_code<WQ>(tile[tx][i], sc[i]);
            }
        }
        __syncthreads();
    }
}

}  // namespace

// ||W_down[:, c]||_2 of every channel c in fp32 (the weight of channel c's
// term in the down projection's linear combination y = sum_c h_c W_down[:, c],
// used by the contribution-ranked selection).  Thread c walks column c of the
// bf16 W_down [d][F]; consecutive threads read consecutive elements.
__global__ void __launch_bounds__(256)
    k_col_norms(const __nv_bfloat16* __restrict__ w_down, float* __restrict__ norms, int d, int F, int Fp) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= Fp) return;
    float ss = 0.0f;
    if (c < F)
        for (int i = 0; i < d; ++i) {
            const float w = __bfloat162float(w_down[(size_t)i * F + c]);
            ss = fmaf(w, w, ss);
        }
    norms[c] = sqrtf(ss);
}

cudaError_t launch_prepare(int d, int F, const __nv_bfloat16* w_gate, const __nv_bfloat16* w_up,
                           const __nv_bfloat16* w_down, uint8_t* codes, __half2* scales,
                           void* gateup, void* down_t, int wq, float* down_norms,
                           cudaStream_t stream) {
    const int Fp = padded_ff(F);
    const int G = d / kGroup;
    k_col_norms<<<(Fp + 255) / 256, 256, 0, stream>>>(w_down, down_norms, d, F, Fp);
    dim3 qgrid((Fp + 127) / 128, G);
    k_quantize_pack<<<qgrid, 128, 0, stream>>>(w_gate, w_up, codes, scales, d, F, Fp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (wq == 1) {
        k_rowq_gateup<1><<<F, 256, 0, stream>>>(w_gate, w_up, static_cast<uint8_t*>(gateup), d);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        k_rowq_down<1><<<(F + 31) / 32, 256, 0, stream>>>(w_down, static_cast<uint8_t*>(down_t),
                                                          static_cast<uint8_t*>(gateup), d, F);
        return cudaGetLastError();
    }
    if (wq == 2) {
        k_rowq_gateup<2><<<F, 256, 0, stream>>>(w_gate, w_up, static_cast<uint8_t*>(gateup), d);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        k_rowq_down<2><<<(F + 31) / 32, 256, 0, stream>>>(w_down, static_cast<uint8_t*>(down_t),
                                                          static_cast<uint8_t*>(gateup), d, F);
        return cudaGetLastError();
    }
    // gate|up interleave: two strided 2-D copies into the [F][2][d] rows
    const size_t row = (size_t)d * sizeof(__nv_bfloat16);
    __nv_bfloat16* gu = static_cast<__nv_bfloat16*>(gateup);
    e = cudaMemcpy2DAsync(gu, 2 * row, w_gate, row, row, F, cudaMemcpyDeviceToDevice, stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpy2DAsync(gu + d, 2 * row, w_up, row, row, F, cudaMemcpyDeviceToDevice, stream);
    if (e != cudaSuccess) return e;
    dim3 tgrid((F + 31) / 32, (d + 31) / 32);
    k_transpose<<<tgrid, 256, 0, stream>>>(w_down, static_cast<__nv_bfloat16*>(down_t), d, F);
    return cudaGetLastError();
}

}  // namespace prox
