// prox_gather.cu -- Stage 2 of "Prox" (Abstract: the selected channels are
// computed exactly, so all three projections run sparse), i.e. Eq. (1) of
// the PrunePath page restricted to the channel list idx:
//     g_c = W_gate[c] . x,  u_c = W_up[c] . x,  h_c = silu(g_c) u_c,
//     y  += h_c * W_down[:, c]          for c in idx
// With idx = NULL and k = d_ff the same kernel is the dense FFN baseline.
//
// One persistent CTA per SM takes a contiguous run of idx.  For each
// channel a producer warp issues two bulk copies (TMA): the interleaved
// gate|up row pair (4 d bytes) and the W_down^T row (2 d bytes), into a
// ring of stages in shared memory.  16 consumer warps own fixed 8-element
// slices of d (x stays in registers), compute the gate/up partial dots for a
// batch of channels, reduce them across the CTA once per batch, form h in
// fp32, and accumulate h * W_down^T rows into a per-thread fp32 slice of y.
// At the end every CTA adds its y slice with vector atomics (y is zeroed by
// the caller's earlier kernel).
#include "prox_internal.cuh"

namespace prox {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;
constexpr int kMaxBatch = 4;
constexpr int kMaxStages = 8;
constexpr int kMaxChanPerCta = 256;
constexpr int kSmemBudget = 220 * 1024;
constexpr int kGroupRowsMin = 128;  // d_model step

struct GatherParams {
    const __nv_bfloat16* gateup;
    const __nv_bfloat16* down_t;
    const uint16_t* x;
    const int32_t* idx;
    float* y;
    float* h_out;
    float2* acc_zero;
    int* status;
    int acc_n, k, d, nst, batch;
    long long limit_ns;
    int inject_stall;
};

struct GatherCtl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    int last_issued[kMaxStages];
    int chan[kMaxChanPerCta];
    float red[2][kConsumerWarps][2 * kMaxBatch];
    int abort;
};

__host__ __device__ inline size_t stage_bytes(int d) { return (size_t)6 * d; }

int stages_for(int d) {
    int nst = (int)((kSmemBudget - sizeof(GatherCtl)) / stage_bytes(d));
    return nst > kMaxStages ? kMaxStages : nst;
}

// acc += sum_e a_e * b_e over 8 bf16 pairs (bf16 x bf16 -> fp32 products)
__device__ __forceinline__ float dot8_bf16(const uint4 a, const uint4 b, float acc) {
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
            "mov.b32 {al, ah}, %1;\n\t"
            "mov.b32 {bl, bh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, al, bl, %0;\n\t"
            "fma.rn.f32.bf16 %0, ah, bh, %0;\n\t}"
            : "+f"(acc)
            : "r"(av[t]), "r"(bv[t]));
    }
    return acc;
}

template <int CPT>
__global__ void __launch_bounds__(kThreads, 1) k_gather_ffn(const GatherParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    GatherCtl& ctl = *reinterpret_cast<GatherCtl*>(smem_raw);
    uint8_t* stages = smem_raw + ((sizeof(GatherCtl) + 127) / 128) * 128;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int p0 = (int)((long long)blockIdx.x * p.k / gridDim.x);
    const int p1 = (int)((long long)(blockIdx.x + 1) * p.k / gridDim.x);
    const int n = p1 - p0;
    const size_t sbytes = stage_bytes(p.d);
    const int nchunk = p.d / 8;  // 16-byte chunks per row

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nst; ++s) {
            mbar_init(&ctl.full[s], 1);
            mbar_init(&ctl.empty[s], kConsumerWarps);
            ctl.last_issued[s] = -1;
        }
        ctl.abort = 0;
        fence_mbar_init();
    }
    if (p.acc_zero) {  // ready the proxy accumulators for the next call
        for (int i = blockIdx.x * kThreads + threadIdx.x; i < p.acc_n; i += gridDim.x * kThreads)
            p.acc_zero[i] = make_float2(0.0f, 0.0f);
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        for (int i = lane; i < n; i += 32) ctl.chan[i] = p.idx ? p.idx[p0 + i] : p0 + i;
        __syncwarp();
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            for (int i = 0; i < n; ++i) {
                const int s = i % p.nst;
                if (i >= p.nst &&
                    !mbar_wait_bounded(&ctl.empty[s], ((i / p.nst) - 1) & 1, p.limit_ns, &ctl.abort)) {
                    ctl.abort = 1;
                    record_status(p.status, PROX_ERR_TIMEOUT);
                    break;
                }
                if (p.inject_stall && i == 0) continue;  // fault-injection test hook
                const int c = ctl.chan[i];
                uint8_t* st = stages + (size_t)s * sbytes;
                mbar_arrive_expect_tx(&ctl.full[s], (uint32_t)sbytes);
                ctl.last_issued[s] = i;
                bulk_g2s(st, p.gateup + (size_t)c * 2 * p.d, (uint32_t)(4 * p.d), &ctl.full[s], pol);
                bulk_g2s(st + 4 * p.d, p.down_t + (size_t)c * p.d, (uint32_t)(2 * p.d), &ctl.full[s],
                         pol);
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int t = threadIdx.x;
        uint4 xr[CPT];
        float yp[CPT][8];
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
            const int ch = t + q * kConsumers;
            xr[q] = ch < nchunk ? __ldg(reinterpret_cast<const uint4*>(p.x) + ch) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int e = 0; e < 8; ++e) yp[q][e] = 0.0f;
        }
        int buf = 0;
        for (int b0 = 0; b0 < n; b0 += p.batch) {
            const int nb = min(p.batch, n - b0);
            float part[2 * kMaxBatch];
#pragma unroll
            for (int v = 0; v < 2 * kMaxBatch; ++v) part[v] = 0.0f;
            bool ok = true;
#pragma unroll
            for (int bi = 0; bi < kMaxBatch; ++bi) {
                if (bi < nb && ok) {
                    const int i = b0 + bi, s = i % p.nst;
                    bool got = true;
                    if (lane == 0)
                        got = mbar_wait_bounded(&ctl.full[s], (i / p.nst) & 1, p.limit_ns, &ctl.abort);
                    got = __shfl_sync(0xffffffffu, got, 0);
                    if (!got) {
                        ok = false;
                        if (lane == 0) {
                            ctl.abort = 1;
                            record_status(p.status, PROX_ERR_TIMEOUT);
                        }
                    } else {
                        const uint8_t* st = stages + (size_t)s * sbytes;
#pragma unroll
                        for (int q = 0; q < CPT; ++q) {
                            const int ch = t + q * kConsumers;
                            if (ch < nchunk) {
                                const uint4 gw = *reinterpret_cast<const uint4*>(st + (size_t)ch * 16);
                                const uint4 uw = *reinterpret_cast<const uint4*>(st + 2 * p.d + (size_t)ch * 16);
                                part[bi] = dot8_bf16(gw, xr[q], part[bi]);
                                part[kMaxBatch + bi] = dot8_bf16(uw, xr[q], part[kMaxBatch + bi]);
                            }
                        }
                    }
                }
            }
            // reduce the 8 partials across the warp: after the butterfly, lanes
            // 4v..4v+3 hold the warp sum of value v
            float v4[4], v2[2], v1;
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const bool up = lane & 16;
                const float send = up ? part[a] : part[a + 4];
                const float keep = up ? part[a + 4] : part[a];
                v4[a] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
            }
#pragma unroll
            for (int a = 0; a < 2; ++a) {
                const bool up = lane & 8;
                const float send = up ? v4[a] : v4[a + 2];
                const float keep = up ? v4[a + 2] : v4[a];
                v2[a] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
            }
            {
                const bool up = lane & 4;
                const float send = up ? v2[0] : v2[1];
                const float keep = up ? v2[1] : v2[0];
                v1 = keep + __shfl_xor_sync(0xffffffffu, send, 4);
            }
            v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
            v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
            if ((lane & 3) == 0) ctl.red[buf][warp][lane >> 2] = v1;
            named_barrier_sync(1, kConsumers);
            if (ctl.abort) break;  // uniform: read after the barrier
            float tot = 0.0f;
            if (lane < 2 * kMaxBatch) {
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) tot += ctl.red[buf][w][lane];
            }
            const float u = __shfl_sync(0xffffffffu, tot, (lane + kMaxBatch) & 31);
            float h = 0.0f;
            if (lane < nb) h = tot / (1.0f + expf(-tot)) * u;  // silu(g) * u
            if (p.h_out && warp == 0 && lane < nb) p.h_out[p0 + b0 + lane] = h;
            float hb[kMaxBatch];
#pragma unroll
            for (int bi = 0; bi < kMaxBatch; ++bi) hb[bi] = __shfl_sync(0xffffffffu, h, bi);
#pragma unroll
            for (int bi = 0; bi < kMaxBatch; ++bi) {
                if (bi < nb) {
                    const int s = (b0 + bi) % p.nst;
                    const uint8_t* st = stages + (size_t)s * sbytes + 4 * p.d;
#pragma unroll
                    for (int q = 0; q < CPT; ++q) {
                        const int ch = t + q * kConsumers;
                        if (ch < nchunk) {
                            const uint4 dw = *reinterpret_cast<const uint4*>(st + (size_t)ch * 16);
                            const uint32_t dv[4] = {dw.x, dw.y, dw.z, dw.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                yp[q][2 * e] = fmaf(hb[bi], __uint_as_float(dv[e] << 16), yp[q][2 * e]);
                                yp[q][2 * e + 1] = fmaf(hb[bi], __uint_as_float(dv[e] & 0xffff0000u), yp[q][2 * e + 1]);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                for (int bi = 0; bi < nb; ++bi) mbar_arrive(&ctl.empty[(b0 + bi) % p.nst]);
            buf ^= 1;
        }
        if (!ctl.abort) {
#pragma unroll
            for (int q = 0; q < CPT; ++q) {
                const int ch = t + q * kConsumers;
                if (ch < nchunk && n > 0) {
                    float* dst = p.y + (size_t)ch * 8;
                    red_add_v4(dst, yp[q][0], yp[q][1], yp[q][2], yp[q][3]);
                    red_add_v4(dst + 4, yp[q][4], yp[q][5], yp[q][6], yp[q][7]);
                }
            }
        }
    }
    __syncthreads();
    if (ctl.abort && threadIdx.x == 0) {
        // drain copies still in flight into this CTA's stages before leaving
        for (int s = 0; s < p.nst; ++s) {
            const int i = ctl.last_issued[s];
            if (i >= 0) mbar_wait_bounded(&ctl.full[s], (i / p.nst) & 1, p.limit_ns, nullptr);
        }
    }
}

size_t smem_bytes(int d, int nst) {
    return ((sizeof(GatherCtl) + 127) / 128) * 128 + (size_t)nst * stage_bytes(d);
}

template <int CPT>
cudaError_t launch_cpt(const GatherParams& p, int grid, cudaStream_t stream) {
    k_gather_ffn<CPT><<<grid, kThreads, smem_bytes(p.d, p.nst), stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t gather_configure(int d) {
    // One attribute for every d: the largest ring any supported d uses.
    (void)d;
    size_t bytes = 0;
    for (int dd = kGroupRowsMin; dd <= kMaxDModel; dd += kGroupRowsMin) {
        const size_t b = smem_bytes(dd, stages_for(dd));
        if (b > bytes) bytes = b;
    }
    cudaError_t e = cudaFuncSetAttribute(k_gather_ffn<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gather_ffn<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_gather_ffn<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    return e;
}

cudaError_t launch_gather_ffn(const __nv_bfloat16* gateup, const __nv_bfloat16* down_t,
                              const uint16_t* x, const int32_t* idx, int k, int d, float* y,
                              float* h_out, float2* acc_zero, int acc_n, int* status,
                              int num_sms, long long wait_limit_ns, int inject_stall,
                              cudaStream_t stream) {
    GatherParams p;
    p.gateup = gateup;
    p.down_t = down_t;
    p.x = x;
    p.idx = idx;
    p.y = y;
    p.h_out = h_out;
    p.acc_zero = acc_zero;
    p.status = status;
    p.acc_n = acc_n;
    p.k = k;
    p.d = d;
    p.nst = stages_for(d);
    p.batch = p.nst >= 2 * kMaxBatch ? kMaxBatch : (p.nst / 2 > 0 ? p.nst / 2 : 1);
    p.limit_ns = wait_limit_ns;
    p.inject_stall = inject_stall;
    int grid = num_sms < k ? num_sms : k;
    if ((k + grid - 1) / grid > kMaxChanPerCta) grid = (k + kMaxChanPerCta - 1) / kMaxChanPerCta;
    if (grid < 1) grid = 1;
    const int nchunk = d / 8;
    if (nchunk <= kConsumers) return launch_cpt<1>(p, grid, stream);
    if (nchunk <= 2 * kConsumers) return launch_cpt<2>(p, grid, stream);
    return launch_cpt<4>(p, grid, stream);
}

}  // namespace prox
