// prox_select.cu -- the two selection steps of "Prox" (Abstract):
//   * input sparsity: keep the k_x entries of largest |x| (ties -> lower
//     index) as the sparsified input of Stage 1;
//   * the shared channel mask: the k channels with the largest proxy
//     magnitude |silu(g~) u~| (ties -> lower channel).
// Both are exact single-CTA radix selects (prox_select.cuh).
#include "prox_select.cuh"

namespace prox {
namespace {

constexpr int kSelThreads = 1024;

// Input sparsity.  Also zeroes y (the Stage-2 kernel accumulates into it)
// and stores the power-of-two prescale that puts max|x| in [2^14, 2^15),
// so every kept x_j * 2^shift is an exact fp16 (its 8 significant bits fit)
// for the proxy's fp16 x fp16 -> fp32 products.
template <int E>
__global__ void __launch_bounds__(kSelThreads)
k_input_select(const uint16_t* __restrict__ x, int d, int kx, int* __restrict__ meta,
               uint32_t* __restrict__ kept, int32_t* __restrict__ kept_out,
               float* __restrict__ y_zero) {
    __shared__ SelectSmem<kSelThreads> sm;
    __shared__ uint32_t smax[kSelThreads / 32];
    uint32_t key[E];
    uint16_t raw[E];
    const int base = threadIdx.x * E;
    uint32_t mk = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int j = base + e;
        raw[e] = j < d ? x[j] : (uint16_t)0;
        key[e] = raw[e] & 0x7fffu;  // |x| as bf16 bits: order = order of |x|
        mk = max(mk, key[e]);
    }
    if (y_zero)
        for (int i = threadIdx.x; i < d; i += kSelThreads) y_zero[i] = 0.0f;
    mk = __reduce_max_sync(0xffffffffu, mk);
    if ((threadIdx.x & 31) == 0) smax[threadIdx.x >> 5] = mk;
    __syncthreads();
    mk = 0;
    for (int w = 0; w < kSelThreads / 32; ++w) mk = max(mk, smax[w]);
    int shift = 0;
    if (mk != 0) {
        int ex;
        frexpf(__uint_as_float(mk << 16), &ex);  // max|x| in [2^(ex-1), 2^ex)
        shift = 15 - ex;
    }
    if (threadIdx.x == 0) meta[1] = shift;

    uint32_t T, r;
    block_kth_largest<kSelThreads, E>(key, 15, (uint32_t)kx, sm, T, r);
    block_compact_topk<kSelThreads, E>(key, T, r, sm, [&](uint32_t pos, int e) {
        const int j = base + e;
        const float xs = ldexpf(__uint_as_float((uint32_t)raw[e] << 16), shift);
        const uint16_t h = __half_as_ushort(__float2half_rn(xs));
        kept[pos] = ((uint32_t)j << 16) | h;
        if (kept_out) kept_out[pos] = j;
    });
}

// Channel mask from the proxy accumulators (g~, u~).
template <int KPT>
__global__ void __launch_bounds__(kSelThreads)
k_channel_select(const float2* __restrict__ acc, int F, int k, int32_t* __restrict__ idx,
                 float* __restrict__ scores, float* __restrict__ scores_out) {
    __shared__ SelectSmem<kSelThreads> sm;
    uint32_t key[KPT];
    const int base = threadIdx.x * KPT;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
        const int c = base + e;
        key[e] = 0;
        if (c < F) {
            const float2 a = acc[c];
            // |silu(g~) * u~|, silu(z) = z / (1 + e^-z)
            const float sc = fabsf(a.x / (1.0f + expf(-a.x)) * a.y);
            key[e] = __float_as_uint(sc);
            if (scores) scores[c] = sc;
            if (scores_out) scores_out[c] = sc;
        }
    }
    uint32_t T, r;
    block_kth_largest<kSelThreads, KPT>(key, 31, (uint32_t)k, sm, T, r);
    block_compact_topk<kSelThreads, KPT>(key, T, r, sm,
                                         [&](uint32_t pos, int e) { idx[pos] = base + e; });
}

template <int E>
cudaError_t input_select_e(const uint16_t* x, int d, int kx, const Workspace& ws,
                           int32_t* kept_out, float* y_zero, cudaStream_t stream) {
    k_input_select<E><<<1, kSelThreads, 0, stream>>>(x, d, kx, ws.status, ws.kept, kept_out,
                                                     y_zero);
    return cudaGetLastError();
}

template <int KPT>
cudaError_t channel_select_k(const Workspace& ws, int F, int k, float* scores_out,
                             cudaStream_t stream) {
    k_channel_select<KPT><<<1, kSelThreads, 0, stream>>>(ws.acc, F, k, ws.idx, ws.scores,
                                                         scores_out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_input_select(const uint16_t* x, int d, int kx, const Workspace& ws,
                                int32_t* kept_out, float* y_zero, cudaStream_t stream) {
    const int per = (d + kSelThreads - 1) / kSelThreads;
    if (per <= 1) return input_select_e<1>(x, d, kx, ws, kept_out, y_zero, stream);
    if (per <= 2) return input_select_e<2>(x, d, kx, ws, kept_out, y_zero, stream);
    if (per <= 4) return input_select_e<4>(x, d, kx, ws, kept_out, y_zero, stream);
    if (per <= 8) return input_select_e<8>(x, d, kx, ws, kept_out, y_zero, stream);
    return input_select_e<16>(x, d, kx, ws, kept_out, y_zero, stream);
}

cudaError_t launch_channel_select(const Workspace& ws, int F, int k, float* scores_out,
                                  cudaStream_t stream) {
    const int per = (F + kSelThreads - 1) / kSelThreads;
    if (per <= 1) return channel_select_k<1>(ws, F, k, scores_out, stream);
    if (per <= 2) return channel_select_k<2>(ws, F, k, scores_out, stream);
    if (per <= 4) return channel_select_k<4>(ws, F, k, scores_out, stream);
    if (per <= 8) return channel_select_k<8>(ws, F, k, scores_out, stream);
    if (per <= 16) return channel_select_k<16>(ws, F, k, scores_out, stream);
    return channel_select_k<32>(ws, F, k, scores_out, stream);
}

}  // namespace prox
