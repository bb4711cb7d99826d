// prox_select.cuh -- single-CTA exact top-k by magnitude with the lowest
// index winning ties, emitting the kept indices in ascending order.
//
// Used twice on the Prox hot path ("Prox", Abstract): for the input
// sparsity (top-|x| over d_model entries) and for the shared channel mask
// (top-k of the proxy magnitude over d_ff channels).  Keys are unsigned
// integers whose order equals the order of the magnitudes (|bf16| bit
// patterns, or the bit patterns of non-negative binary32 scores), so the
// selection is an exact radix select: 8-bit digits from the top, one
// shared-memory histogram per digit, then one block scan to place each kept
// element.  Each thread owns KPT consecutive elements, so index order is
// thread order.
#pragma once

#include "prox_internal.cuh"

namespace prox {

template <int NT>
struct SelectSmem {
    uint32_t hist[256];
    uint32_t warp_tot[NT / 32 + 1];
    uint32_t result[2];
};

// Exclusive block scan of one value per thread; also returns the total.
template <int NT>
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, SelectSmem<NT>& sm,
                                                         uint32_t& total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t s = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += t;
    }
    if (lane == 31) sm.warp_tot[wid] = s;
    __syncthreads();
    if (wid == 0) {
        const uint32_t w = lane < NT / 32 ? sm.warp_tot[lane] : 0u;
        uint32_t ws = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, ws, o);
            if (lane >= o) ws += t;
        }
        if (lane < NT / 32) sm.warp_tot[lane] = ws - w;
        if (lane == NT / 32 - 1) sm.warp_tot[NT / 32] = ws;
    }
    __syncthreads();
    const uint32_t excl = sm.warp_tot[wid] + s - v;
    total = sm.warp_tot[NT / 32];
    __syncthreads();
    return excl;
}

// Finds T, the k-th largest key held by the block (1 <= k <= number of
// keys), and r = k - #(keys > T), the number of keys equal to T to keep.
// Keys are < 2^nbits, nbits <= 31.
template <int NT, int KPT>
__device__ __forceinline__ void block_kth_largest(const uint32_t (&key)[KPT], int nbits,
                                                  uint32_t k, SelectSmem<NT>& sm, uint32_t& T,
                                                  uint32_t& r) {
    uint32_t prefix = 0, krem = k;
    int bits_left = nbits;
    bool first = true;
    while (bits_left > 0) {
        const int db = bits_left >= 8 ? 8 : bits_left;
        const int shift = bits_left - db;
        const uint32_t mask = (1u << db) - 1u;
        for (int i = threadIdx.x; i < 256; i += NT) sm.hist[i] = 0;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < KPT; ++e) {
            const uint32_t kk = key[e];
            if (first || (kk >> (shift + db)) == prefix) atomicAdd(&sm.hist[(kk >> shift) & mask], 1u);
        }
        __syncthreads();
        // Suffix counts over the bins: thread t < 256 looks at bin 255 - t.
        const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
        uint32_t v = 0, s = 0;
        if (threadIdx.x < 256) {
            v = sm.hist[255 - threadIdx.x];
            s = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t t = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += t;
            }
            if (lane == 31) sm.warp_tot[wid] = s;
        }
        __syncthreads();
        if (threadIdx.x < 256) {
            for (int w = 0; w < wid; ++w) s += sm.warp_tot[w];
            // s = #candidates with digit >= 255 - t
            if (s >= krem && s - v < krem) {
                sm.result[0] = 255u - threadIdx.x;
                sm.result[1] = krem - (s - v);
            }
        }
        __syncthreads();
        prefix = (prefix << db) | sm.result[0];
        krem = sm.result[1];
        bits_left -= db;
        first = false;
        __syncthreads();
    }
    T = prefix;
    r = krem;
}

// Emits, in ascending index order, the indices whose key is > T plus the
// first r (lowest-index) whose key == T.  Element e of thread t has index
// t * KPT + e.  Calls emit(pos, e) for each kept element of this thread.
template <int NT, int KPT, typename Emit>
__device__ __forceinline__ void block_compact_topk(const uint32_t (&key)[KPT], uint32_t T,
                                                   uint32_t r, SelectSmem<NT>& sm, Emit emit) {
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
        gt += key[e] > T;
        eq += key[e] == T;
    }
    uint32_t total;
    const uint32_t excl = block_exclusive_scan<NT>((eq << 16) | gt, sm, total);
    const uint32_t pe = excl >> 16, pg = excl & 0xffffu;
    uint32_t pos = pg + (pe < r ? pe : r);
    uint32_t tie = pe;
#pragma unroll
    for (int e = 0; e < KPT; ++e) {
        bool keep = key[e] > T;
        if (key[e] == T) {
            keep = tie < r;
            ++tie;
        }
        if (keep) emit(pos++, e);
    }
}

}  // namespace prox
