// prox_fused.cu -- the whole Prox decode step ("Prox: Training-Free FFN
// Activation Sparsity via Approximate Intermediate-Channel Salience in
// LLMs", Abstract) as ONE persistent kernel, one CTA per SM, phases
// separated by bounded grid barriers:
//
//   P0  input sparsity: every CTA selects the k_x entries of largest |x|
//       (ties -> lower index) itself from x (a few KB, L2 resident), so no
//       launch or barrier precedes the proxy stream.
//   P1  proxy GEMV (Stage 1): CTA (tile, slice) streams the int4 proxy rows
//       of its slice of the kept inputs, restricted to its channel tile, with
//       128-bit loads, and writes per-slice partial (g~, u~) sums.
//   --- grid barrier
//   P2  CTA i owns a chunk of channels: sums the slices in a fixed order
//       (deterministic scores), forms |silu(g~) u~| and adds the channels to
//       a global 11-bit histogram of the score bit patterns.
//   --- grid barrier
//   P3  every CTA finishes the exact top-k itself: the histogram gives the
//       bin of the k-th score; two more digit passes over the candidates of
//       that bin (all scores staged in shared memory) give the threshold and
//       the number of ties to keep (lowest channels first).  A block scan
//       places every selected channel in the ascending list; the CTA keeps
//       positions [k i / n, k (i+1) / n).
//   P4  Stage 2 on those channels (Eq. (1) of the PrunePath page restricted
//       to the mask): gate|up rows and W_down^T rows arrive by bulk copies
//       (TMA) into two shared-memory rings; 16 warps own 8-element slices of
//       d_model, form partial dot products, reduce them across warps one
//       batch behind (mbarrier-synchronised), compute h = silu(g) u in fp32
//       and accumulate h * W_down^T into registers; one vector atomic per
//       element adds the CTA's part of y at the end.
//
// The same Stage-2 code, over all channels, is the dense baseline
// (k_dense).  Every wait is bounded: a wait that runs out records
// PROX_ERR_TIMEOUT in the layer's status word, lets copies in flight land
// and leaves the kernel.
#include "prox_internal.cuh"

namespace prox {
namespace {

constexpr int kNT = 576;                 // 18 warps
constexpr int kConsumerWarps = 16;       // Stage-2 consumers
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kGuProducerWarp = 16;
constexpr int kDProducerWarp = 17;
constexpr int kMaxStages = 16;
constexpr int kMaxChan = 512;            // Stage-2 channels per CTA
constexpr int kRing = 8;                 // proxy rows in flight per thread (cp.async ring)
static_assert((kRing & (kRing - 1)) == 0, "ring depth must be a power of two");
constexpr int kHistBins = 2048;
constexpr size_t kSmemLimit = 227 * 1024;
constexpr int kPhaseStamps = 10;

// Phase timestamp (tracing only): thread 0 of the CTA stores %globaltimer.
__device__ __forceinline__ void stamp(uint64_t* ts, int i) {
    if (ts && threadIdx.x == 0) ts[(size_t)blockIdx.x * kPhaseStamps + i] = global_timer_ns();
}

struct Ctl {
    uint64_t gu_full[kMaxStages], gu_empty[kMaxStages];
    uint64_t d_full[kMaxStages], d_empty[kMaxStages];
    int gu_last[kMaxStages], d_last[kMaxStages];
    float h[kMaxChan];
    uint32_t warp_tot[kNT / 32 + 1];
    uint32_t sel[4];
    uint64_t ld_bar[2];  // bulk loads of the proxy scales (P1) and the scores (P3)
    unsigned epoch;
    int abort;
    int chan[kMaxChan];
};

constexpr size_t ctl_bytes() { return (sizeof(Ctl) + 127) / 128 * 128; }
__host__ __device__ constexpr size_t area_budget_dev() { return kSmemLimit - ctl_bytes(); }

struct FusedParams {
    // layer
    const uint8_t* codes;
    const __half2* scales;
    const __nv_bfloat16* gateup;
    const __nv_bfloat16* down_t;
    int d, F, Fp;
    // call
    const uint16_t* x;
    float* y;
    int kx, k;
    // proxy geometry
    int tiles, slices, tile_w;
    // workspace
    int* status;
    unsigned* bar;
    unsigned* epoch;     // number of completed calls on this workspace
    uint32_t* hist;      // [kHistBins]
    float2* part;        // [slices][Fp]
    float* scores;       // [Fp]
    // debug outputs (may be null)
    int32_t* kept_out;
    float* scores_out;
    int32_t* idx_out;
    float* h_out;
    // stage-2 ring geometry
    int n_gu, n_d;
    long long limit_ns;
    int inject;          // 1: the last CTA skips the first grid barrier (test hook)
    uint64_t* ts;        // [gridDim][kPhaseStamps] %globaltimer stamps, or null
};

// ----------------------------------------------------------------- helpers
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_add_release_gpu(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid-wide barrier for co-resident CTAs.  The barrier word counts arrivals
// and is never reset between calls: in call number `epoch` (read by every
// CTA at its start) barrier i (1 or 2) completes when the word reaches
// n * (2 epoch + i).  Arrivals are fire-and-forget release reductions; CTA
// thread 0 polls with acquire loads.  Returns false (and records
// PROX_ERR_TIMEOUT) if the count does not arrive within limit_ns.
__device__ bool grid_barrier(unsigned* bar, unsigned target, int* status, long long limit_ns,
                             Ctl& ctl, bool skip_arrive) {
    __syncthreads();
    if (threadIdx.x == 0) {
        bool ok = !skip_arrive;
        if (ok) {
            red_add_release_gpu(bar, 1u);
            uint64_t t0 = 0;
            for (uint32_t it = 1;; ++it) {
                if ((int)(ld_acquire_gpu(bar) - target) >= 0) break;
                if ((it & 15u) == 0) {
                    const uint64_t now = global_timer_ns();
                    if (t0 == 0) t0 = now;
                    else if ((long long)(now - t0) > limit_ns) {
                        ok = false;
                        break;
                    }
                }
            }
        }
        if (!ok) {
            record_status(status, PROX_ERR_TIMEOUT);
            ctl.abort = 1;
        }
    }
    __syncthreads();
    return ctl.abort == 0;
}

// Given a histogram h[nbins] of digits (nbins a multiple of 128, at most
// 2048) and krem >= 1 with sum(h) >= krem, warp 0 finds the digit b with
// sum(h[b+1..]) < krem <= sum(h[b..]) and stores (b, krem - sum(h[b+1..]))
// in sel[0..1].  Level 1: lane l sums the nbins/32 bins just below
// nbins - l nbins/32 (independent vector loads) and a warp scan finds the
// lane holding the k-th; level 2 spreads that lane's bins over the warp
// (at most two per lane) and scans again.  No data-dependent loop.  Called
// by warp 0 only; the caller synchronises.
template <int NBINS>
__device__ __forceinline__ void select_bin_warp(const uint32_t* h, uint32_t krem, uint32_t* sel) {
    constexpr int PER = NBINS / 32, NQ = PER / 4, PER2 = PER > 32 ? 2 : 1;
    static_assert(NBINS % 128 == 0 && NBINS <= 2048, "bins");
    const int lane = threadIdx.x & 31;
    const int lo = NBINS - (lane + 1) * PER;
    const uint4* hv = reinterpret_cast<const uint4*>(h + lo);
    uint4 w[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) w[q] = hv[q];  // all loads in flight at once
    uint32_t sum = 0;
#pragma unroll
    for (int q = 0; q < NQ; ++q) sum += (w[q].x + w[q].y) + (w[q].z + w[q].w);
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, incl - sum < krem && incl >= krem);
    const int L = hit ? __ffs(hit) - 1 : 0;  // hit != 0 whenever sum(h) >= krem
    const uint32_t above_l = __shfl_sync(0xffffffffu, incl - sum, L);
    const int top = NBINS - L * PER - 1;  // lane L's highest bin
    // level 2: lane l takes bins top - PER2 l and (PER2 = 2) top - 2 l - 1
    const int b0 = top - lane * PER2;
    uint32_t v0 = 0, v1 = 0;
    if (lane * PER2 < PER) v0 = h[b0];
    if (PER2 == 2 && lane * 2 + 1 < PER) v1 = h[b0 - 1];
    const uint32_t s2 = v0 + v1;
    uint32_t incl2 = s2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl2, o);
        if (lane >= o) incl2 += t;
    }
    const uint32_t above2 = above_l + incl2 - s2;
    if (above2 < krem && above2 + s2 >= krem) {
        if (above2 + v0 >= krem) {
            sel[0] = (uint32_t)b0;
            sel[1] = krem - above2;
        } else {
            sel[0] = (uint32_t)(b0 - 1);
            sel[1] = krem - above2 - v0;
        }
    }
}

// Exclusive scan of one value per thread over the block (warp shuffles, one
// barrier); also returns the block total.  Uses ctl.warp_tot.
// Barrier over the first NT threads: __syncthreads for the whole block,
// named barrier 1 for a prefix of warps.
template <int NT>
__device__ __forceinline__ void group_sync() {
    if (NT == kNT) __syncthreads();
    else named_barrier_sync(1, NT);
}

template <int NT = kNT>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, Ctl& ctl, uint32_t& total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t s = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += t;
    }
    if (lane == 31) ctl.warp_tot[wid] = s;
    group_sync<NT>();
    uint32_t wp = 0, tt = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        const uint32_t x = ctl.warp_tot[w];
        wp += w < wid ? x : 0u;
        tt += x;
    }
    total = tt;
    return wp + s - v;
}

// Exact top-k over n keys in shared memory (thread t owns the contiguous
// keys [t kpt, (t+1) kpt), kpt <= 64), ties to the lower index, in three
// radix digits: d1 = key >> s1 from a histogram h1 already built, then the
// next digits over the thread's own candidates only (the keys in the
// selected d1 bin, tracked in a bit mask), so only the first pass touches
// every key.  Produces T (the k-th key) and r (ties at T to keep) in
// ctl.sel[0..1], and for this thread: the number of selected keys before
// its range (in ascending index order) and a candidate mask.
struct TopkPlan {
    int s1, n1;        // digit-1 shift and histogram size (h1)
    int s2, n2;        // digit-2 shift and bins (h2), digit 3 = key & (n3 - 1)
    int n3;
};

template <int NT, typename KeyFn>
__device__ __forceinline__ void topk_digits(const TopkPlan& pl, int n, int kpt, uint32_t k,
                                            KeyFn key, uint32_t* h1, uint32_t* h2, uint32_t* h3,
                                            Ctl& ctl, uint32_t& T, uint32_t& r, uint32_t& pos0,
                                            uint32_t& ties_before, uint32_t& nsel) {
    const int wid = threadIdx.x >> 5;
    const int i0 = threadIdx.x * kpt;
    // digit 1 from h1
    if (wid == 0) {
        if (pl.n1 == 2048) select_bin_warp<2048>(h1, k, ctl.sel);
        else select_bin_warp<256>(h1, k, ctl.sel);
    }
    group_sync<NT>();
    const uint32_t b1 = ctl.sel[0], k1 = ctl.sel[1];
    uint32_t gt1 = 0;
    uint64_t cmask = 0;
    for (int e = 0; e < kpt; ++e) {
        const int i = i0 + e;
        if (i < n) {
            const uint32_t d1 = key(i) >> pl.s1;
            gt1 += d1 > b1;
            cmask |= (uint64_t)(d1 == b1) << e;
        }
    }
    for (uint64_t m = cmask; m; m &= m - 1)
        atomicAdd(&h2[(key(i0 + __ffsll((long long)m) - 1) >> pl.s2) & (pl.n2 - 1)], 1u);
    group_sync<NT>();
    if (wid == 0) {
        if (pl.n2 == 2048) select_bin_warp<2048>(h2, k1, ctl.sel);
        else select_bin_warp<128>(h2, k1, ctl.sel);
    }
    group_sync<NT>();
    const uint32_t b12 = (b1 << (pl.s1 - pl.s2)) | ctl.sel[0], k2 = ctl.sel[1];
    if (pl.n3 > 1) {
        for (uint64_t m = cmask; m; m &= m - 1) {
            const uint32_t kk = key(i0 + __ffsll((long long)m) - 1);
            if ((kk >> pl.s2) == b12) atomicAdd(&h3[kk & (pl.n3 - 1)], 1u);
        }
        group_sync<NT>();
        if (wid == 0) select_bin_warp<512>(h3, k2, ctl.sel);
        group_sync<NT>();
        T = (b12 << pl.s2) | ctl.sel[0];
        r = ctl.sel[1];
    } else {
        T = b12;
        r = k2;
    }
    // per-thread counts from the sure keys and the thread's own candidates
    uint32_t gt = gt1, eq = 0;
    for (uint64_t m = cmask; m; m &= m - 1) {
        const uint32_t kk = key(i0 + __ffsll((long long)m) - 1);
        gt += kk > T;
        eq += kk == T;
    }
    uint32_t tot;
    const uint32_t ex = block_excl_scan<NT>(gt | (eq << 16), ctl, tot);
    ties_before = ex >> 16;
    pos0 = (ex & 0xffffu) + min(ties_before, r);  // selected keys before this range
    nsel = gt + (ties_before < r ? min(eq, r - ties_before) : 0u);
}

// Bulk prefetch of global memory into L2 (no shared-memory destination).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// fp16 bits of x * 2^shift for a bf16 x (exact whenever the result is a
// normal fp16; the same rounding as ldexpf followed by __float2half_rn).
__device__ __forceinline__ uint16_t scaled_fp16(uint16_t xb, int shift) {
    const uint32_t f = (uint32_t)xb << 16;
    const int e = (int)((f >> 23) & 0xffu);
    float v;
    if (e != 0 && e + shift > 0 && e + shift < 255)
        v = __uint_as_float(f + ((uint32_t)shift << 23));  // exact power-of-two scaling
    else
        v = ldexpf(__uint_as_float(f), shift);
    return __half_as_ushort(__float2half_rn(v));
}

// --------------------------------------------------------------- proxy math
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
    return d;
}

__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
    __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hfma2_bits(uint32_t a, uint32_t b, uint32_t c) {
    __half2 r = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b),
                        *reinterpret_cast<__half2*>(&c));
    return *reinterpret_cast<uint32_t*>(&r);
}

// acc0 += q.lo * x, acc1 += q.hi * x  (fp16 x fp16 -> fp32, one rounding each)
__device__ __forceinline__ void fma_f32_f16x2(float& acc0, float& acc1, uint32_t q, uint16_t x) {
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "fma.rn.f32.f16 %0, l, %3, %0;\n\t"
        "fma.rn.f32.f16 %1, h, %3, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "r"(q), "h"(x));
}

// One 32-bit word of proxy codes = 4 channels (byte = gate | up << 4, each
// nibble offset-binary q + 8).  The nibbles become exact fp16 integers with
// one LOP3 and one packed HSUB2/HFMA2 per two channels.
__device__ __forceinline__ void proxy_mac_word(uint32_t w, uint16_t xh, float* ag, float* au) {
    constexpr uint32_t kLo = 0x000F000Fu, kHi = 0x00F000F0u, kMagic = 0x64006400u;
    constexpr uint32_t kBias = 0x64086408u;      // (1032, 1032)
    constexpr uint32_t kSixteenth = 0x2C002C00u; // (1/16, 1/16)
    constexpr uint32_t kHiBias = 0xD480D480u;    // (-72, -72)
    const uint32_t w8 = w >> 8;
    const uint32_t g02 = hsub2_bits(lop3_and_or(w, kLo, kMagic), kBias);
    const uint32_t g13 = hsub2_bits(lop3_and_or(w8, kLo, kMagic), kBias);
    const uint32_t u02 = hfma2_bits(lop3_and_or(w, kHi, kMagic), kSixteenth, kHiBias);
    const uint32_t u13 = hfma2_bits(lop3_and_or(w8, kHi, kMagic), kSixteenth, kHiBias);
    fma_f32_f16x2(ag[0], ag[2], g02, xh);
    fma_f32_f16x2(ag[1], ag[3], g13, xh);
    fma_f32_f16x2(au[0], au[2], u02, xh);
    fma_f32_f16x2(au[1], au[3], u13, xh);
}

// 16-byte global -> shared copy that bypasses L1 (cp.async), L2 policy hint.
__device__ __forceinline__ void cp_async_16(void* dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)),
                 "l"(src), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Waits until at most N of this thread's cp.async groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- stage 2
// acc += sum over 8 bf16 pairs of a_e * b_e in fp32 (bf16 -> fp32 is exact)
__device__ __forceinline__ float dot8_bf16(const uint4 a, const uint4 b, float acc) {
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        acc = fmaf(__uint_as_float(av[t] << 16), __uint_as_float(bv[t] << 16), acc);
        acc = fmaf(__uint_as_float(av[t] & 0xffff0000u), __uint_as_float(bv[t] & 0xffff0000u), acc);
    }
    return acc;
}

struct Stage2Args {
    const __nv_bfloat16* gateup;
    const __nv_bfloat16* down_t;
    const uint16_t* x;
    float* y;
    float* h_out;   // [k], written at pos0 + i (may be null)
    int* status;
    int d, n_gu, n_d, pos0;
    long long limit_ns;
    uint64_t* ts;   // [gridDim][kPhaseStamps] or null
};

// Waits (every lane polls) for the phase; on a timeout records the status
// and raises the CTA's abort flag.  Returns false on timeout or abort.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, long long limit_ns,
                                          Ctl& ctl, int* status) {
    const bool got = mbar_wait_bounded(bar, parity, limit_ns, &ctl.abort);
    if (!got && (threadIdx.x & 31) == 0) {
        ctl.abort = 1;
        record_status(status, PROX_ERR_TIMEOUT);
    }
    return __all_sync(0xffffffffu, got);
}

// Stage 2 over the n channels ctl.chan[0..n).  Shared area `area`: x as bf16
// (2 d bytes), then n_gu gate|up stages (4 d bytes each), then n_d W_down^T
// stages (2 d bytes each).
//   pass A: warp w < n_gu computes g_c, u_c for channels i = w, w + n_gu, ...
//           over the whole gate|up row (warp-local reduction),
//           h_c = silu(g_c) u_c;
//   pass B: every consumer thread owns 8-element slices of d and adds
//           h_c * W_down^T[c, slice] for all channels in order.
// The W_down^T ring fills during pass A.
template <int CPT>
__device__ void stage2(const Stage2Args& a, Ctl& ctl, uint8_t* area, int n) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = a.d, n_gu = a.n_gu, n_d = a.n_d;
    const size_t gu_bytes = (size_t)4 * d, d_bytes = (size_t)2 * d;
    uint16_t* xs = reinterpret_cast<uint16_t*>(area);
    uint8_t* gu_ring = area + (size_t)2 * d;
    uint8_t* d_ring = gu_ring + (size_t)n_gu * gu_bytes;
    const int nchunk = d / 8;  // 16-byte chunks per row

    stamp(a.ts, 6);
    if (threadIdx.x == 0) {
        for (int s = 0; s < n_gu; ++s) {
            mbar_init(&ctl.gu_full[s], 1);
            mbar_init(&ctl.gu_empty[s], 1);
            ctl.gu_last[s] = -1;
        }
        for (int s = 0; s < n_d; ++s) {
            mbar_init(&ctl.d_full[s], 1);
            mbar_init(&ctl.d_empty[s], kConsumerWarps);
            ctl.d_last[s] = -1;
        }
        fence_mbar_init();
    }
    __syncthreads();  // the producers start before the consumers fetch x

    if (warp == kGuProducerWarp || warp == kDProducerWarp) {
        if (lane == 0) {
            const bool gu = warp == kGuProducerWarp;
            const int ns = gu ? n_gu : n_d;
            const size_t sb = gu ? gu_bytes : d_bytes;
            uint64_t* full = gu ? ctl.gu_full : ctl.d_full;
            uint64_t* empty = gu ? ctl.gu_empty : ctl.d_empty;
            int* last = gu ? ctl.gu_last : ctl.d_last;
            uint8_t* base = gu ? gu_ring : d_ring;
            const uint8_t* src = gu ? reinterpret_cast<const uint8_t*>(a.gateup)
                                    : reinterpret_cast<const uint8_t*>(a.down_t);
            const uint64_t pol = policy_evict_first();
            for (int i = 0; i < n; ++i) {
                const int s = i % ns;
                if (i >= ns &&
                    !mbar_wait_bounded(&empty[s], ((i / ns) - 1) & 1, a.limit_ns, &ctl.abort)) {
                    ctl.abort = 1;
                    record_status(a.status, PROX_ERR_TIMEOUT);
                    break;
                }
                if (ctl.abort) break;
                const int c = ctl.chan[i];
                last[s] = i;
                mbar_arrive_expect_tx(&full[s], (uint32_t)sb);
                bulk_g2s(base + (size_t)s * sb, src + (size_t)c * sb, (uint32_t)sb, &full[s], pol);
            }
        }
    } else {
        for (int i = threadIdx.x; i < nchunk; i += kConsumers)
            reinterpret_cast<uint4*>(xs)[i] = __ldg(reinterpret_cast<const uint4*>(a.x) + i);
        named_barrier_sync(1, kConsumers);
        // ------------------------------------------------ pass A: h per channel
        // Warp w < n_gu owns gate|up slot w and takes channels w, w + n_gu, ...
        // Each slot's uses are consumed in order by one warp, so a parity wait
        // can never be taken for a phase two uses ahead (which would pass at
        // once and release the slot while its copy is still in flight).
        bool ok = true;
        for (int i = warp; warp < n_gu && i < n && ok; i += n_gu) {
            const int s = warp;
            ok = warp_wait(&ctl.gu_full[s], (i / n_gu) & 1, a.limit_ns, ctl, a.status);
            if (!ok) break;
            if (i == 0 && lane == 0 && a.ts)
                a.ts[(size_t)blockIdx.x * kPhaseStamps + 7] = global_timer_ns();
            const uint4* gr = reinterpret_cast<const uint4*>(gu_ring + (size_t)s * gu_bytes);
            const uint4* ur = gr + nchunk;
            const uint4* xv = reinterpret_cast<const uint4*>(xs);
            float g = 0.0f, u = 0.0f;
            for (int ch = lane; ch < nchunk; ch += 32) {
                const uint4 xw = xv[ch];
                g = dot8_bf16(gr[ch], xw, g);
                u = dot8_bf16(ur[ch], xw, u);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                g += __shfl_xor_sync(0xffffffffu, g, o);
                u += __shfl_xor_sync(0xffffffffu, u, o);
            }
            if (lane == 0) {
                mbar_arrive(&ctl.gu_empty[s]);
                const float h = g / (1.0f + expf(-g)) * u;  // silu(g) * u
                ctl.h[i] = h;
                if (a.h_out) a.h_out[a.pos0 + i] = h;
            }
        }
        named_barrier_sync(1, kConsumers);
        // ------------------------------------------------ pass B: y += h W_down^T
        const int t = threadIdx.x;
        float yp[CPT][8];
#pragma unroll
        for (int q = 0; q < CPT; ++q)
#pragma unroll
            for (int e = 0; e < 8; ++e) yp[q][e] = 0.0f;
        ok = ok && !ctl.abort;
        for (int i = 0; i < n && ok; ++i) {
            const int s = i % n_d;
            ok = warp_wait(&ctl.d_full[s], (i / n_d) & 1, a.limit_ns, ctl, a.status);
            if (!ok) break;
            const float hv = ctl.h[i];
            const uint8_t* st = d_ring + (size_t)s * d_bytes;
#pragma unroll
            for (int q = 0; q < CPT; ++q) {
                const int ch = t + q * kConsumers;
                if (ch < nchunk) {
                    const uint4 dw = *reinterpret_cast<const uint4*>(st + (size_t)ch * 16);
                    const uint32_t dv[4] = {dw.x, dw.y, dw.z, dw.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        yp[q][2 * e] = fmaf(hv, __uint_as_float(dv[e] << 16), yp[q][2 * e]);
                        yp[q][2 * e + 1] = fmaf(hv, __uint_as_float(dv[e] & 0xffff0000u), yp[q][2 * e + 1]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.d_empty[s]);
        }
        if (warp == 0 && lane == 0 && a.ts)
            a.ts[(size_t)blockIdx.x * kPhaseStamps + 8] = global_timer_ns();
        if (ok && !ctl.abort && n > 0) {
#pragma unroll
            for (int q = 0; q < CPT; ++q) {
                const int ch = t + q * kConsumers;
                if (ch < nchunk) {
                    float* dst = a.y + (size_t)ch * 8;
                    red_add_v4(dst, yp[q][0], yp[q][1], yp[q][2], yp[q][3]);
                    red_add_v4(dst + 4, yp[q][4], yp[q][5], yp[q][6], yp[q][7]);
                }
            }
        }
    }
    __syncthreads();
    stamp(a.ts, 9);
    if (ctl.abort && threadIdx.x == 0) {
        // let the copies still in flight into this CTA's rings land before leaving
        for (int s = 0; s < n_gu; ++s)
            if (ctl.gu_last[s] >= 0)
                mbar_wait_bounded(&ctl.gu_full[s], (ctl.gu_last[s] / n_gu) & 1, a.limit_ns, nullptr);
        for (int s = 0; s < n_d; ++s)
            if (ctl.d_last[s] >= 0)
                mbar_wait_bounded(&ctl.d_full[s], (ctl.d_last[s] / n_d) & 1, a.limit_ns, nullptr);
    }
}

// P3: every CTA finishes the exact top-k of the scores itself (threads
// 0..NT-1; NT a multiple of 32, named barrier 1): the global digit-1
// histogram and all scores arrive by bulk copy, three radix digits over each
// thread's own candidates give the threshold, one block scan the positions;
// the CTA keeps the channels at positions [p0, p1) in ctl.chan.  On a
// timeout it raises ctl.abort (after letting the copy land).
template <int NT>
__device__ __forceinline__ void select_channels(const FusedParams& p, Ctl& ctl, uint8_t* area,
                                                int b, int nb, int p0, int p1) {
    const int tid = threadIdx.x, lane = tid & 31;
    const int F = p.F, Fp = p.Fp;
    // area: global histogram copy [2048] | digit-2 histogram [2048] |
    // digit-3 histogram [512] | scores [Fp]
    uint32_t* h1 = reinterpret_cast<uint32_t*>(area);
    uint32_t* h2 = h1 + kHistBins;
    uint32_t* h3 = h2 + kHistBins;
    float* sc = reinterpret_cast<float*>(h3 + 512);
    if (tid == 0) {
        asm volatile("fence.proxy.async.global;" ::: "memory");
        const uint64_t pol = policy_evict_first();
        mbar_arrive_expect_tx(&ctl.ld_bar[1], (uint32_t)(kHistBins * 4 + Fp * 4));
        bulk_g2s(h1, p.hist, kHistBins * 4, &ctl.ld_bar[1], pol);
        bulk_g2s(sc, p.scores, (uint32_t)(Fp * 4), &ctl.ld_bar[1], pol);
    }
    for (int i = tid; i < kHistBins + 512; i += NT) h2[i] = 0u;
    if (!mbar_wait_bounded(&ctl.ld_bar[1], 0, p.limit_ns, &ctl.abort) && lane == 0) {
        ctl.abort = 1;
        record_status(p.status, PROX_ERR_TIMEOUT);
    }
    named_barrier_sync(1, NT);
    if (ctl.abort) {
        // let the copy land (bounded) before the shared memory is released
        if (tid == 0) mbar_wait_bounded(&ctl.ld_bar[1], 0, p.limit_ns, nullptr);
        return;
    }
    // exact top-k of the score bit patterns: digits of 11, 11 and 9 bits;
    // thread t owns the channels [t kpf, (t+1) kpf)
    const int kpf = (F + NT - 1) / NT;  // <= 64
    const int ci0 = tid * kpf;
    auto skey = [&](int i) { return __float_as_uint(sc[i]); };
    uint32_t T, r, cpos, cties, cn;
    {
        const TopkPlan pls{20, 2048, 9, 2048, 512};
        topk_digits<NT>(pls, F, kpf, (uint32_t)p.k, skey, h1, h2, h3, ctl, T, r, cpos, cties, cn);
    }
    // only the threads whose positions [cpos, cpos + cn) meet [p0, p1) emit
    if (cn && (int)(cpos + cn) > p0 && (int)cpos < p1) {
        uint32_t pos = cpos, tie = cties;
        for (int e = 0; e < kpf; ++e) {
            const int c = ci0 + e;
            if (c < F) {
                const uint32_t kk = skey(c);
                bool keep = kk > T;
                if (kk == T) {
                    keep = tie < r;
                    ++tie;
                }
                if (keep) {
                    if ((int)pos >= p0 && (int)pos < p1) ctl.chan[pos - p0] = c;
                    ++pos;
                }
            }
        }
    }
    // the debug channel list: every selected channel, by its owner thread
    if (p.idx_out && b == 0 && cn) {
        uint32_t pos = cpos, tie = cties;
        for (int e = 0; e < kpf; ++e) {
            const int c = ci0 + e;
            if (c < F) {
                const uint32_t kk = skey(c);
                bool keep = kk > T;
                if (kk == T) {
                    keep = tie < r;
                    ++tie;
                }
                if (keep) p.idx_out[pos++] = c;
            }
        }
    }
    (void)nb;
}

// ------------------------------------------------------------ fused kernel
template <int CPT>
__global__ void __launch_bounds__(kNT, 1) k_prox_fused(const FusedParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Ctl& ctl = *reinterpret_cast<Ctl*>(smem_raw);
    uint8_t* area = smem_raw + ctl_bytes();  // phase-dependent union
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nb = gridDim.x, b = blockIdx.x;
    const int d = p.d, F = p.F, Fp = p.Fp;
    stamp(p.ts, 0);
    if (tid == 0) {
        ctl.abort = 0;
        ctl.epoch = *reinterpret_cast<volatile unsigned*>(p.epoch);
        mbar_init(&ctl.ld_bar[0], 1);
        mbar_init(&ctl.ld_bar[1], 1);
        fence_mbar_init();
    }

    // ------------------------------------------------ P0: input sparsity
    // area: x bf16 [d] | kept u32 [d] | histograms u32 [1024] | P1 tables
    // Warp w takes the x entries [w Lx, (w+1) Lx), lane-consecutive.
    uint16_t* xs = reinterpret_cast<uint16_t*>(area);
    uint32_t* kept = reinterpret_cast<uint32_t*>(area + (size_t)2 * d);
    uint32_t* hA = kept + d;
    for (int i = tid; i < d / 8; i += kNT)
        reinterpret_cast<uint4*>(xs)[i] = __ldg(reinterpret_cast<const uint4*>(p.x) + i);
    for (int i = tid; i < 384; i += kNT) hA[i] = 0u;
    if (b == 0) {
        for (int i = tid; i < d; i += kNT) p.y[i] = 0.0f;
        for (int i = tid; i < kHistBins; i += kNT) p.hist[i] = 0u;
    }
    __syncthreads();
    // exact top-k_x of |x| (15-bit keys): digit 1 = exponent (bits 14..7),
    // digit 2 = the 7 mantissa bits; thread t owns [t kpx, (t+1) kpx)
    const int kpx = (d + kNT - 1) / kNT;
    const int xi0 = tid * kpx;
    auto xkey = [&](int i) { return (uint32_t)(xs[i] & 0x7fffu); };
    {
        uint32_t mk = 0;
        for (int e = 0; e < kpx; ++e) {
            const int i = xi0 + e;
            if (i < d) {
                const uint32_t kk = xkey(i);
                mk = max(mk, kk);
                atomicAdd(&hA[kk >> 7], 1u);
            }
        }
        mk = __reduce_max_sync(0xffffffffu, mk);
        if (lane == 0) ctl.warp_tot[wid] = mk;
    }
    __syncthreads();
    if (tid == 0) {  // power-of-two prescale: max|x| * 2^shift in [2^14, 2^15)
        uint32_t mk = 0;
        for (int w = 0; w < kNT / 32; ++w) mk = max(mk, ctl.warp_tot[w]);
        int sh = 0;
        if (mk != 0) {
            int ex;
            frexpf(__uint_as_float(mk << 16), &ex);  // max|x| in [2^(ex-1), 2^ex)
            sh = 15 - ex;
        }
        ctl.sel[2] = (uint32_t)sh;
    }
    uint32_t xT, xr, xpos, xties, xn;
    {
        const TopkPlan plx{7, 256, 0, 128, 1};
        topk_digits<kNT>(plx, d, kpx, (uint32_t)p.kx, xkey, hA, hA + 256, nullptr, ctl, xT, xr,
                         xpos, xties, xn);
    }
    const int shift = (int)ctl.sel[2];
    if (xn) {
        uint32_t pos = xpos, tie = xties;
        for (int e = 0; e < kpx; ++e) {
            const int j = xi0 + e;
            if (j < d) {
                const uint32_t kk = xkey(j);
                bool keep = kk > xT;
                if (kk == xT) {
                    keep = tie < xr;
                    ++tie;
                }
                if (keep) {
                    kept[pos] = ((uint32_t)j << 16) | scaled_fp16(xs[j], shift);
                    if (b == 0 && p.kept_out) p.kept_out[pos] = j;
                    ++pos;
                }
            }
        }
    }
    __syncthreads();
    stamp(p.ts, 1);

    // ------------------------------------------------ P1: proxy partials
    if (b < p.tiles * p.slices) {
        const int tile = b % p.tiles, slice = b / p.tiles;
        const int W = p.tile_w;
        const int c0 = tile * W;
        const int width = min(W, Fp - c0);
        const int tpr = W / 16;
        const int R = kNT / tpr;
        const int rl = tid / tpr, cu = tid % tpr;
        const bool active = rl < R && cu * 16 < width;
        const int r0 = (int)((long long)slice * p.kx / p.slices);
        const int r1 = (int)((long long)(slice + 1) * p.kx / p.slices);
        // row-lane rl takes the contiguous kept rows [q_beg, q_end)
        const int m = (r1 - r0 + R - 1) / R;
        const int q_beg = min(r1, r0 + rl * m), q_end = min(r1, q_beg + m);
        // running totals, [R][16][tpr] float2: channel cu * 16 + t of row-lane
        // rl at (rl * 16 + t) * tpr + cu, so a warp's lanes (consecutive cu)
        // touch consecutive 8-byte words
        float2* tot = reinterpret_cast<float2*>(hA + 1024);
        // per-thread ring of proxy row segments in flight, [kRing][kNT]
        uint4* ring = reinterpret_cast<uint4*>(tot + (size_t)R * 16 * tpr);
        uint8_t* after_ring = reinterpret_cast<uint8_t*>(ring + (size_t)kRing * kNT);
        const size_t room = area_budget_dev() - (size_t)(after_ring - area);
        // the slice's fp16 scale pairs, [g - g_lo][W], loaded by bulk copies
        int g_lo = 0, ng = 0;
        if (r1 > r0) {
            g_lo = (int)(kept[r0] >> 23);
            ng = (int)(kept[r1 - 1] >> 23) - g_lo + 1;
        }
        uint32_t* ssc = reinterpret_cast<uint32_t*>(after_ring);
        const bool smem_scales = ng > 0 && (size_t)ng * W * 4 <= room;
        if (tid == 0 && smem_scales) {
            const uint64_t pol = policy_evict_first();
            mbar_arrive_expect_tx(&ctl.ld_bar[0], (uint32_t)(ng * width * 4));
            for (int g = 0; g < ng; ++g)
                bulk_g2s(ssc + (size_t)g * W, p.scales + (size_t)(g_lo + g) * Fp + c0,
                         (uint32_t)(width * 4), &ctl.ld_bar[0], pol);
        }
        if (active)
            for (int t = 0; t < 16; ++t) tot[((size_t)rl * 16 + t) * tpr + cu] = make_float2(0.0f, 0.0f);
        float ag[16], au[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) ag[t] = au[t] = 0.0f;
        int cur_g = -1;
        bool scales_in = false;
        auto flush = [&]() {
            if (cur_g < 0) return;
            const uint4* src;
            if (smem_scales) {
                if (!scales_in) {
                    if (!mbar_wait_bounded(&ctl.ld_bar[0], 0, p.limit_ns, &ctl.abort)) {
                        ctl.abort = 1;
                        record_status(p.status, PROX_ERR_TIMEOUT);
                    }
                    scales_in = true;
                }
                src = reinterpret_cast<const uint4*>(ssc + (size_t)(cur_g - g_lo) * W + cu * 16);
            } else {
                src = reinterpret_cast<const uint4*>(p.scales + (size_t)cur_g * Fp + c0 + cu * 16);
            }
            float2* dst = tot + (size_t)rl * 16 * tpr + cu;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 s4 = src[v];
                const uint32_t sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = 4 * v + e;
                    const float2 s2 = __half22float2(*reinterpret_cast<const __half2*>(&sv[e]));
                    float2 o = dst[(size_t)t * tpr];
                    o.x = fmaf(s2.x, ag[t], o.x);
                    o.y = fmaf(s2.y, au[t], o.y);
                    dst[(size_t)t * tpr] = o;
                    ag[t] = 0.0f;
                    au[t] = 0.0f;
                }
            }
        };
        if (active && q_beg < q_end) {
            // kRing rows in flight per thread through a cp.async ring in
            // shared memory (slot s of thread t at ring[s * kNT + t]); each
            // thread reads only its own slots, so no block synchronisation.
            // With tpr a multiple of 16 the row, and kept[q], is uniform
            // across each half-warp.  One row per iteration keeps the loop
            // body (and its instruction footprint) small.
            const uint64_t pol = policy_evict_first();
            const uint8_t* colbase = p.codes + c0 + cu * 16;
            uint4* my = ring + tid;
#pragma unroll
            for (int u = 0; u < kRing; ++u) {
                const int q = q_beg + u;
                if (q < q_end)
                    cp_async_16(my + (size_t)u * kNT, colbase + (size_t)(kept[q] >> 16) * Fp, pol);
                cp_async_commit();
            }
            int s = 0;
#pragma unroll 1
            for (int q = q_beg; q < q_end; ++q) {
                cp_async_wait_group<kRing - 1>();  // row q has landed
                const uint4 w = my[(size_t)s * kNT];
                const uint32_t kp = kept[q];
                const int qn = q + kRing;
                if (qn < q_end)
                    cp_async_16(my + (size_t)s * kNT, colbase + (size_t)(kept[qn] >> 16) * Fp, pol);
                cp_async_commit();
                s = (s + 1) & (kRing - 1);
                const int g = (int)(kp >> 23);  // j / 128
                if (g != cur_g) {
                    flush();
                    cur_g = g;
                }
                const uint16_t xh = (uint16_t)(kp & 0xffffu);
                proxy_mac_word(w.x, xh, &ag[0], &au[0]);
                proxy_mac_word(w.y, xh, &ag[4], &au[4]);
                proxy_mac_word(w.z, xh, &ag[8], &au[8]);
                proxy_mac_word(w.w, xh, &ag[12], &au[12]);
            }
            cp_async_wait_group<0>();
            flush();
        }
        // the scale copy must have landed before this shared memory is reused
        if (smem_scales && !scales_in)
            if (!mbar_wait_bounded(&ctl.ld_bar[0], 0, p.limit_ns, &ctl.abort)) {
                ctl.abort = 1;
                record_status(p.status, PROX_ERR_TIMEOUT);
            }
        __syncthreads();
        float2* out = p.part + (size_t)slice * Fp + c0;
        // thread e sums channel (e % tpr) * 16 + e / tpr over the row-lanes:
        // consecutive threads read consecutive 8-byte words
        for (int e = tid; e < 16 * tpr; e += kNT) {
            const int cu_ = e % tpr, t_ = e / tpr;
            const int cl = cu_ * 16 + t_;
            if (cl < width) {
                float g = 0.0f, u = 0.0f;
                for (int r = 0; r < R; ++r) {
                    const float2 v = tot[((size_t)r * 16 + t_) * tpr + cu_];
                    g += v.x;
                    u += v.y;
                }
                out[cl] = make_float2(ldexpf(g, -shift), ldexpf(u, -shift));
            }
        }
    }
    stamp(p.ts, 2);
    const unsigned ep = ctl.epoch;
    if (!grid_barrier(p.bar, (unsigned)nb * (2u * ep + 1u), p.status, p.limit_ns, ctl,
                      p.inject == 1 && b == nb - 1))
        return;
    stamp(p.ts, 3);

    // ------------------------------------------------ P2: scores + histogram
    const int cb0 = (int)((long long)F * b / nb), cb1 = (int)((long long)F * (b + 1) / nb);
    float* lsc = ctl.h;  // this chunk's scores (ctl.h is Stage 2's, free until then)
    {
        for (int c00 = cb0; c00 < cb1; c00 += kNT) {
            const int c = c00 + tid;
            const bool act = c < cb1;
            uint32_t key = 0;
            if (act) {
                float2 v[kMaxSlices];
#pragma unroll
                for (int sl = 0; sl < kMaxSlices; ++sl)
                    if (sl < p.slices) v[sl] = __ldcg(p.part + (size_t)sl * Fp + c);
                float g = 0.0f, u = 0.0f;
#pragma unroll
                for (int sl = 0; sl < kMaxSlices; ++sl)
                    if (sl < p.slices) {
                        g += v[sl].x;
                        u += v[sl].y;
                    }
                // |silu(g~) * u~|, silu(z) = z / (1 + e^-z)
                const float sc = fabsf(g / (1.0f + expf(-g)) * u);
                p.scores[c] = sc;
                if (p.scores_out) p.scores_out[c] = sc;
                lsc[c - cb0] = sc;
                key = __float_as_uint(sc);
            }
            // one reduction per distinct bin in the warp
            const unsigned am = __ballot_sync(0xffffffffu, act);
            if (act) {
                const unsigned peers = __match_any_sync(am, key >> 20);
                if (lane == __ffs(peers) - 1)
                    asm volatile("red.global.add.u32 [%0], %1;" ::"l"(p.hist + (key >> 20)),
                                 "r"((uint32_t)__popc(peers))
                                 : "memory");
            }
        }
    }
    stamp(p.ts, 4);
    // Grid barrier 2, then the channel selection (P3) on warps 0..15 while
    // warp 17 prefetches: the channels ranked in the top 90% of this chunk's
    // expected share of the mask are almost surely selected, and their
    // Stage-2 rows (gate|up, W_down^T) are prefetched into L2 so that HBM
    // streams during the selection.  A wrong guess costs bandwidth only.  The
    // prefetch warp stays off the selection's barriers (bulk prefetches can
    // stall their issuing thread while the copy engine's queue is full).
    constexpr int kSel = 512;  // threads of warps 0..15
    const int p0 = (int)((long long)p.k * b / nb), p1 = (int)((long long)p.k * (b + 1) / nb);
    const int n_mine = p1 - p0;
    __syncthreads();
    if (tid == 0) red_add_release_gpu(p.bar, 1u);
    if (wid == kNT / 32 - 1) {
        const int nch = cb1 - cb0;
        const int m = (int)(0.9 * (double)p.k * nch / F);
        for (int i = lane; i < nch; i += 32) {
            const float mine = lsc[i];
            int rank = 0;
            for (int j = 0; j < nch; ++j) {
                const float o = lsc[j];
                rank += (o > mine) || (o == mine && j < i);
            }
            if (rank < m) {
                const int c = cb0 + i;
                prefetch_l2(p.gateup + (size_t)c * 2 * d, (uint32_t)(4 * d));
                prefetch_l2(p.down_t + (size_t)c * d, (uint32_t)(2 * d));
            }
        }
    } else if (tid < kSel) {
        if (tid == 0) {
            const unsigned target = (unsigned)nb * (2u * ep + 2u);
            bool ok = true;
            uint64_t t0 = 0;
            for (uint32_t it = 1;; ++it) {
                if ((int)(ld_acquire_gpu(p.bar) - target) >= 0) break;
                if ((it & 15u) == 0) {
                    const uint64_t now = global_timer_ns();
                    if (t0 == 0) t0 = now;
                    else if ((long long)(now - t0) > p.limit_ns) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok) {
                record_status(p.status, PROX_ERR_TIMEOUT);
                ctl.abort = 1;
            } else if (b == 0) {
                *reinterpret_cast<volatile unsigned*>(p.epoch) = ep + 1u;
            }
        }
        named_barrier_sync(1, kSel);
        if (!ctl.abort) {
            stamp(p.ts, 5);
            select_channels<kSel>(p, ctl, area, b, nb, p0, p1);
        }
    }
    __syncthreads();  // channel list ready, prefetches issued
    if (ctl.abort) return;

    // ------------------------------------------------ P4: stage 2
    Stage2Args a;
    a.gateup = p.gateup;
    a.down_t = p.down_t;
    a.x = p.x;
    a.y = p.y;
    a.h_out = p.h_out;
    a.status = p.status;
    a.d = d;
    a.n_gu = p.n_gu;
    a.n_d = p.n_d;
    a.pos0 = (int)((long long)p.k * b / nb);
    a.limit_ns = p.limit_ns;
    a.ts = p.ts;
    stage2<CPT>(a, ctl, area, n_mine);
}

// Dense baseline: Stage 2 over every channel, CTA i taking [F i/n, F (i+1)/n).
template <int CPT>
__global__ void __launch_bounds__(kNT, 1) k_dense(const Stage2Args a0, int F) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Ctl& ctl = *reinterpret_cast<Ctl*>(smem_raw);
    uint8_t* area = smem_raw + ctl_bytes();
    if (threadIdx.x == 0) ctl.abort = 0;
    const int c0 = (int)((long long)F * blockIdx.x / gridDim.x);
    const int c1 = (int)((long long)F * (blockIdx.x + 1) / gridDim.x);
    for (int i = threadIdx.x; i < c1 - c0; i += kNT) ctl.chan[i] = c0 + i;
    __syncthreads();
    Stage2Args a = a0;
    a.pos0 = c0;
    stamp(a.ts, 0);
    stage2<CPT>(a, ctl, area, c1 - c0);
}

// ------------------------------------------------------------ host side
struct Ring {
    int n_gu, n_d;
};

size_t area_budget() { return kSmemLimit - ctl_bytes(); }

// Stage-2 rings: x (2 d bytes) plus as many gate|up (4 d) and W_down^T
// (2 d) stages as fit, about 60% of the ring bytes for gate|up.
Ring ring_for(int d) {
    const size_t budget = area_budget() - (size_t)2 * d;
    const size_t gu = (size_t)4 * d, dd = (size_t)2 * d;
    Ring r{0, 0};
    int best = -1;
    for (int ng = 1; ng <= kMaxStages; ++ng)
        for (int nd = 1; nd <= kMaxStages; ++nd) {
            if ((size_t)ng * gu + (size_t)nd * dd > budget) continue;
            const int bytes = ng * 4 + nd * 2;   // in units of d bytes
            const int score = 4 * bytes - abs(ng * 4 - 3 * nd * 2);  // prefer full, balanced
            if (score > best) {
                best = score;
                r = {ng, nd};
            }
        }
    return r;
}

size_t ring_bytes(int d, const Ring& r) {
    return (size_t)2 * d + (size_t)r.n_gu * 4 * d + (size_t)r.n_d * 2 * d;
}

template <typename K>
cudaError_t set_smem(K kern) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
}

}  // namespace

ProxyGeom proxy_geometry(int F, int kx, int num_blocks) {
    // Tiles of W = 256, 512 or 1024 channels (a half-warp, a warp or two
    // warps per proxy row), T tiles x S slices <= blocks; minimise the
    // bytes of the busiest CTA, then prefer fewer slices (less partial
    // traffic).
    const int Fp = padded_ff(F);
    ProxyGeom best{1, 1, 1024};
    long long best_cost = -1;
    for (int W : {256, 512, 1024}) {
        const int T = (Fp + W - 1) / W;
        if (T > num_blocks) continue;
        int S = num_blocks / T;
        if (S > kMaxSlices) S = kMaxSlices;
        if (S > kx) S = kx;
        if (S < 1) S = 1;
        const long long cost = (long long)min(W, Fp) * ((kx + S - 1) / S);
        if (best_cost < 0 || cost < best_cost || (cost == best_cost && S < best.slices)) {
            best_cost = cost;
            best = {T, S, W};
        }
    }
    return best;
}

cudaError_t fused_configure() {
    cudaError_t e = set_smem(k_prox_fused<1>);
    if (e == cudaSuccess) e = set_smem(k_prox_fused<2>);
    if (e == cudaSuccess) e = set_smem(k_prox_fused<4>);
    if (e == cudaSuccess) e = set_smem(k_dense<1>);
    if (e == cudaSuccess) e = set_smem(k_dense<2>);
    if (e == cudaSuccess) e = set_smem(k_dense<4>);
    return e;
}

size_t fused_smem_bytes() { return kSmemLimit; }

int fused_threads() { return kNT; }

int fused_max_chan() { return kMaxChan; }

bool fused_fits(int d, int F) {
    // P0: x (2 d) + kept list (4 d) + histogram; P1 adds the [R][W] partial
    // table (at most 8 * 16 * kNT bytes); P3: histogram + F scores; P4: rings.
    const size_t p01 = (size_t)6 * d + 4096 + (size_t)8 * 16 * kNT + (size_t)16 * kRing * kNT;
    const size_t p3 = (size_t)(2 * kHistBins + 512) * 4 + (size_t)4 * padded_ff(F);
    const Ring r = ring_for(d);
    return p01 <= area_budget() && p3 <= area_budget() && ring_bytes(d, r) <= area_budget() &&
           r.n_gu >= 1 && r.n_d >= 1;
}

cudaError_t launch_fused(const FusedLaunch& L, cudaStream_t stream) {
    FusedParams p;
    p.codes = L.codes;
    p.scales = L.scales;
    p.gateup = L.gateup;
    p.down_t = L.down_t;
    p.d = L.d;
    p.F = L.F;
    p.Fp = padded_ff(L.F);
    p.x = L.x;
    p.y = L.y;
    p.kx = L.kx;
    p.k = L.k;
    const ProxyGeom geo = proxy_geometry(L.F, L.kx, L.num_blocks);
    p.tiles = geo.tiles;
    p.slices = geo.slices;
    p.tile_w = geo.tile_w;
    p.status = L.ws->status;
    p.bar = L.ws->bar;
    p.epoch = L.ws->bar + 1;
    p.hist = L.ws->hist;
    p.part = L.ws->part;
    p.scores = L.ws->scores;
    p.kept_out = L.kept_out;
    p.scores_out = L.scores_out;
    p.idx_out = L.idx_out;
    p.h_out = L.h_out;
    const Ring r = ring_for(L.d);
    p.n_gu = r.n_gu;
    p.n_d = r.n_d;
    p.limit_ns = L.limit_ns;
    p.inject = L.inject;
    p.ts = L.ts;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.num_blocks);
    cfg.blockDim = dim3(kNT);
    cfg.dynamicSmemBytes = kSmemLimit;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int nchunk = L.d / 8;
    if (nchunk <= kConsumers) return cudaLaunchKernelEx(&cfg, k_prox_fused<1>, p);
    if (nchunk <= 2 * kConsumers) return cudaLaunchKernelEx(&cfg, k_prox_fused<2>, p);
    return cudaLaunchKernelEx(&cfg, k_prox_fused<4>, p);
}

cudaError_t launch_dense(const __nv_bfloat16* gateup, const __nv_bfloat16* down_t,
                         const uint16_t* x, int d, int F, float* y, int* status, int num_blocks,
                         long long limit_ns, uint64_t* ts, cudaStream_t stream) {
    Stage2Args a;
    a.gateup = gateup;
    a.down_t = down_t;
    a.x = x;
    a.y = y;
    a.h_out = nullptr;
    a.status = status;
    a.d = d;
    const Ring r = ring_for(d);
    a.n_gu = r.n_gu;
    a.n_d = r.n_d;
    a.pos0 = 0;
    a.limit_ns = limit_ns;
    a.ts = ts;
    const int nchunk = d / 8;
    if (nchunk <= kConsumers) k_dense<1><<<num_blocks, kNT, kSmemLimit, stream>>>(a, F);
    else if (nchunk <= 2 * kConsumers) k_dense<2><<<num_blocks, kNT, kSmemLimit, stream>>>(a, F);
    else k_dense<4><<<num_blocks, kNT, kSmemLimit, stream>>>(a, F);
    return cudaGetLastError();
}

}  // namespace prox
