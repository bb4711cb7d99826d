// prox_prepare.cu -- one-off per-layer preparation (not on the timed path).
//
// "Prox" (Abstract): Stage 1 reads quantized proxy copies of W_gate and W_up;
// Stage 2 reads the selected gate/up rows and down-projection columns.  This
// file builds:
//   * the int4 group-128 symmetric proxy, packed input-dim-major so that one
//     kept input dimension is one contiguous row of d_ff bytes;
//   * the channel-interleaved gate|up rows and the channel-major W_down^T.
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

}  // namespace

cudaError_t launch_prepare(int d, int F, const __nv_bfloat16* w_gate, const __nv_bfloat16* w_up,
                           const __nv_bfloat16* w_down, uint8_t* codes, __half2* scales,
                           __nv_bfloat16* gateup, __nv_bfloat16* down_t, cudaStream_t stream) {
    const int Fp = padded_ff(F);
    const int G = d / kGroup;
    dim3 qgrid((Fp + 127) / 128, G);
    k_quantize_pack<<<qgrid, 128, 0, stream>>>(w_gate, w_up, codes, scales, d, F, Fp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // gate|up interleave: two strided 2-D copies into the [F][2][d] rows
    const size_t row = (size_t)d * sizeof(__nv_bfloat16);
    e = cudaMemcpy2DAsync(gateup, 2 * row, w_gate, row, row, F, cudaMemcpyDeviceToDevice, stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpy2DAsync(gateup + d, 2 * row, w_up, row, row, F, cudaMemcpyDeviceToDevice, stream);
    if (e != cudaSuccess) return e;
    dim3 tgrid((F + 31) / 32, (d + 31) / 32);
    k_transpose<<<tgrid, 256, 0, stream>>>(w_down, down_t, d, F);
    return cudaGetLastError();
}

}  // namespace prox
