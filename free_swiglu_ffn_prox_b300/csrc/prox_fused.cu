// prox_fused.cu -- the whole Prox decode step ("Prox: Training-Free FFN
// Activation Sparsity via Approximate Intermediate-Channel Salience in
// LLMs", Abstract) as ONE persistent kernel, one CTA per SM:
//
//   P0  input sparsity: every CTA selects the k_x entries of largest |x|
//       (ties -> lower index) itself from x (a few KB, L2 resident), so no
//       launch or barrier precedes the proxy stream.
//   P1  proxy GEMV (Stage 1): CTA (tile, slice) streams the int4 proxy rows
//       of its slice of the kept inputs, restricted to its channel tile,
//       through a per-thread cp.async ring, and writes per-slice partial
//       (g~, u~) sums.
//   --- grid barrier 1
//   P2  CTA b owns the channel chunk [cb0, cb1) (chunk starts on multiples of
//       4 channels, ~F/n wide): sums the slices in a fixed order
//       (deterministic scores), forms |silu(g~) u~| (times ||W_down[:, c]||
//       for the contribution signal; block sums for a block mask), publishes
//       every channel's score key (the fp32 bits) in channel order and adds
//       the chunk to a global histogram of the keys' top 11 bits.
//   --- grid barrier 2
//   P3a every CTA finds the exact k-th key itself: it stages all keys from L2
//       into shared memory while it selects the digit-1 bin from the global
//       histogram, then resolves digits 2 (bits 19..9) and 3 (bits 8..0)
//       over that bin's candidates with loads-only passes that build
//       per-thread bit masks; ties go to the lower channel.  A block scan
//       gives every selected channel its position in channel order, and CTA
//       b takes the positions [k b / n, k (b+1) / n) as its Stage-2 items
//       (an even split: every CTA moves the same bytes).
//   P3b Stage 2 (Eq. (1) of the PrunePath page restricted to the mask):
//       gate|up rows arrive by bulk copies (TMA) into a shared-memory ring
//       (bytes in flight capped), and so do bf16 W_down^T rows; for int8 or
//       int4 rows every pass-B thread streams its own W_down^T slices with
//       cp.async.  Pass-A warps form h = silu(W_gate x) (W_up x) per item
//       (one warp per row), pass-B warps own slices of d_model and
//       accumulate h * W_down^T; one vector atomic per element adds the
//       CTA's part of y at the end.
//   Stage-2 rows are bf16 (WQ = 0), or int8 (1) or int4 (2) codes with one
//   fp32 scale per row: the codes are decoded exactly to fp32 and the scales
//   are applied to g, u and h.
//
// The same step also runs
//   * in a layer stack, several steps in one launch (k_prox_stack), each
//     later layer forming its x from the previous layer's x and y in P0;
//   * mask-only, for a batch over the union of its tokens' masks: after P3a
//     each CTA records its share of the token's mask and skips Stage 2, with
//     one token per launch or a group of CTAs per token (k_prox_masks).
// The same Stage-2 code over all channels is the dense baseline (k_dense).
// Every wait is bounded: a wait that runs out records PROX_ERR_TIMEOUT in
// the layer's status word, lets copies in flight land and leaves the kernel.
#include "prox_internal.cuh"

namespace prox {
namespace {

constexpr int kNT = 608;                  // 19 warps
constexpr int kPassAWarps = 8;            // warps 0..7: gate|up dot products
constexpr int kPassBWarp0 = 8;            // warps 8..15: y += h W_down^T
constexpr int kPassBWarps = 8;
constexpr int kPassB = 32 * kPassBWarps;
constexpr int kGuProducerWarp = 16;
constexpr int kDProducerWarp = 17;
constexpr int kSelectorWarp = 18;
constexpr int kMaxStages = 16;
// 8-element chunks of d per pass-B thread (the kernels' CPT)
__host__ __device__ constexpr int chunks_per_thread(int d) {
    return d / 8 <= kPassB ? 1 : d / 8 <= 2 * kPassB ? 2 : d / 8 <= 4 * kPassB ? 4 : 8;
}
// Codes: bytes of one item's W_down^T slices over all pass-B threads in the
// self-streamed slots (CPT chunks of 8 (int8) or 4 (int4) bytes each).
__host__ __device__ constexpr size_t self_item_bytes(int d, int wq) {
    return (size_t)chunks_per_thread(d) * (wq == 2 ? 4 : 8) * kPassB;
}
constexpr size_t kGuRingBytes = 112 * 1024;   // gate|up bytes in flight per SM (bf16)
constexpr size_t kGuRingBytesQ = 136 * 1024;  // ... (int8 rows: 16 stages at d = 4096; int4)
constexpr size_t kDRingBytes = 48 * 1024;     // W_down^T bytes in flight per SM
constexpr int kMaxItems = 512;            // Stage-2 items per CTA
constexpr int kMaxChunk = 256;            // channels per CTA chunk
constexpr int kMaxBlocks = kMaxGrid;
constexpr int kRing = 16;                 // proxy rows in flight per thread (cp.async ring)
static_assert(kRing >= 8, "the running-total table reuses the ring (16 x 8 bytes per thread)");
static_assert((kRing & (kRing - 1)) == 0, "ring depth must be a power of two");
constexpr int kHistBins = 2048;
constexpr int kXGroups = 3;               // 8-element x groups per thread: d <= 8 * 3 * kNT
static_assert(kHistBins <= kHistWords, "histogram words");
constexpr size_t kSmemLimit = 227 * 1024;
constexpr int kPhaseStamps = 16;

// Phase timestamp (tracing only): thread 0 of the CTA stores %globaltimer.
__device__ __forceinline__ void stamp(uint64_t* ts, int i) {
    if (ts && threadIdx.x == 0) ts[(size_t)blockIdx.x * kPhaseStamps + i] = global_timer_ns();
}

// The same from whichever single thread calls it.
__device__ __forceinline__ void stamp_here(uint64_t* ts, int i) {
    if (ts) ts[(size_t)blockIdx.x * kPhaseStamps + i] = global_timer_ns();
}

struct FusedParams {
    // layer
    const uint8_t* codes;
    const __half2* scales;
    const uint8_t* gateup;  // Stage-2 rows: bf16, or int8 / int4 codes with scales
    const uint8_t* down_t;
    int wq;                 // Stage-2 row format: 0 bf16, 1 int8, 2 int4
    int d, F, Fp;
    // call
    const uint16_t* x;
    float* y;
    int kx, k;
    // block-granular mask: channels per block (a power of two, 4..256; chunk
    // starts are multiples of it) whose summed score ranks the whole block;
    // 0: the per-channel mask
    int bw;
    const float* dnorm;      // contribution-ranked selection: ||W_down[:, c]|| (null: |h~_c|)
    // optional stack glue in front of the step: x = bf16(RMSNorm(x_prev + y_prev))
    const uint16_t* x_prev;  // null: x is given
    const float* y_prev;
    uint16_t* x_out;         // the normalised x, written by CTA 0 (may be null)
    float eps;
    // proxy geometry
    int tiles, slices, tile_w;
    // workspace
    int* status;
    unsigned* bar;       // [0] grid-barrier arrival count, [1] grid barriers completed
                         // on this workspace (control block; a group launch: its word)
    unsigned* epoch;     // grid barriers completed on this workspace (bar + 1)
    uint32_t* hist;      // [kHistWords]: histogram of the score keys' top 11 bits
    float2* part;        // [slices][Fp]
    uint32_t* skey;      // [Fp] every channel's score key (the fp32 score's bits), channel order
    int* idx_list;       // [Fp] debug: the selected channels, ascending
    float* hch;          // [Fp] debug: h per channel
    // debug outputs (may be null)
    int32_t* kept_out;
    float* scores_out;
    int debug;           // write idx_list and hch
    // stage-2 geometry: n_gu gate|up stages consumed by n_a pass-A warps
    // (n_a divides n_gu); n_d W_down^T stages (bf16), or for codes the items
    // each pass-B thread streams ahead (8, 4 or 2)
    int n_gu, n_d, n_a;
    long long limit_ns;
    int inject;          // 1: the last CTA withholds its grid-barrier arrival (test hook)
    uint64_t* ts;        // [gridDim][kPhaseStamps] %globaltimer stamps, or null
    uint32_t* member;    // mask only: per channel the bits of the tokens whose mask holds it
    int token;
    int gsize;           // > 0: the grid is split into groups of gsize CTAs, one token each
};

struct Ctl {
    uint64_t gu_full[kMaxStages], gu_empty[kMaxStages];
    uint64_t d_full[kMaxStages], d_empty[kMaxStages];
    uint64_t done_bar;               // every warp is through its Stage-2 role
    uint64_t ld_bar;                 // bulk load of the proxy scales (P1)
    uint64_t key_ld;                 // bulk load of every channel's score key
    int gu_last[kMaxStages], d_last[kMaxStages];
    float h[kMaxItems];              // h of each item
    int item[kMaxItems];             // channel of each item
    uint8_t hready[kMaxItems];       // h[i] written by pass A
    float lsc[kMaxChunk];            // scores of this CTA's chunk
    __align__(16) uint32_t warp_tot[(kNT / 32 + 4) / 4 * 4];  // per-warp totals, read as uint4
    uint32_t sel[4];
    unsigned epoch;
    int abort;
    int n_items;
    FusedParams sp;                  // the current layer's parameters (stack launch)
};

constexpr size_t ctl_bytes() { return (sizeof(Ctl) + 127) / 128 * 128; }
__host__ __device__ constexpr size_t area_budget_dev() { return kSmemLimit - ctl_bytes(); }


// First channel of chunk b (F <= 32768 and b <= 256, so F b fits 32 bits;
// a 64-bit division costs hundreds of instructions on the GPU).
__host__ __device__ __forceinline__ int chunk_begin(int F, int b, int nb) {
    return (int)((unsigned)F * (unsigned)b / (unsigned)nb);
}

// First channel of CTA b's chunk in the fused kernel: chunk starts are
// multiples of al channels (al = 4, so per-chunk arrays copy in 16-byte
// pieces, or the block width of a block-granular mask, so every chunk holds
// whole blocks); the last chunk ends at F.
__host__ __device__ __forceinline__ int chunk_lo(int F, int b, int nb, int al) {
    const int c = al * chunk_begin((F + al - 1) / al, b, nb);
    return c < F ? c : F;
}

__host__ __device__ __forceinline__ int chunk_align(int bw) { return bw > 0 ? bw : 4; }

// ----------------------------------------------------------------- helpers
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
// and is never reset between calls: `target` is n times the number of the
// barrier (the callers count the barriers completed on the workspace before
// the launch, read by every CTA at its start).  Arrivals are fire-and-forget
// release reductions; CTA thread 0 polls with acquire loads.  Returns false
// (and records PROX_ERR_TIMEOUT) if the count does not arrive within
// limit_ns.
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
    // all warp totals at once (independent 16-byte loads), then sums in registers
    constexpr int NV = (NT / 32 + 3) / 4;
    uint4 wt[NV];
#pragma unroll
    for (int q = 0; q < NV; ++q) wt[q] = reinterpret_cast<const uint4*>(ctl.warp_tot)[q];
    uint32_t wp = 0, tt = 0;
#pragma unroll
    for (int q = 0; q < NV; ++q) {
        const uint32_t x4[4] = {wt[q].x, wt[q].y, wt[q].z, wt[q].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int w = 4 * q + e;
            if (w < NT / 32) {
                wp += w < wid ? x4[e] : 0u;
                tt += x4[e];
            }
        }
    }
    total = tt;
    return wp + s - v;
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
// acc += a * x  (fp16 x fp16 -> fp32, one rounding)
__device__ __forceinline__ void fma_f32_f16(float& acc, uint16_t a, uint16_t x) {
    asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc) : "h"(a), "h"(x));
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
// nibble offset-binary n = q + 8).  A single AND per two channels leaves each
// nibble in the mantissa of an fp16 half with a zero exponent field: the
// exact subnormal n 2^-24 (gate nibbles, bits 0-3 and 16-19) or 16 n 2^-24 =
// n 2^-20 (up nibbles, bits 4-7 and 20-23); the word shifted by 8 gives the
// other two channels.  The fp16 x fp16 -> fp32 products are exact, the group
// sums are sum n x scaled by 2^-24 / 2^-20, and the flush removes the offset
// with sum q x = sum n x - 8 sum x (one FMA per channel, exact whenever the
// sums fit in fp32).
__device__ __forceinline__ void proxy_mac_word(uint32_t w, uint16_t xh, float* ag, float* au) {
    const uint32_t w8 = w >> 8;
    fma_f32_f16x2(ag[0], ag[2], w & 0x000F000Fu, xh);
    fma_f32_f16x2(ag[1], ag[3], w8 & 0x000F000Fu, xh);
    fma_f32_f16x2(au[0], au[2], w & 0x00F000F0u, xh);
    fma_f32_f16x2(au[1], au[3], w8 & 0x00F000F0u, xh);
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

// 4- or 8-byte global -> shared copy (cp.async through L1), L2 policy hint.
template <int B>
__device__ __forceinline__ void cp_async_small(void* dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], %2, %3;" ::"r"(smem_u32(dst)),
                 "l"(src), "n"(B), "l"(pol)
                 : "memory");
}

// ---------------------------------------------------------------- stage 2

// int8 weights: a word of four two's-complement codes, flipped to offset
// binary (w ^ 0x80808080), gives code e as the exact float 2^23 + (q + 128)
// by placing its byte under the exponent of 2^23 (one PRMT); subtracting
// 2^23 + 128 leaves q exactly.  Codes e and e + 1 come as a pair, with one
// packed subtraction.
__device__ __forceinline__ float2 q8_pair(uint32_t wo, int e) {
    const float2 b = make_float2(__uint_as_float(__byte_perm(wo, 0x4Bu, 0x4550u | (unsigned)e)),
                                 __uint_as_float(__byte_perm(wo, 0x4Bu, 0x4550u | (unsigned)(e + 1))));
    return __fadd2_rn(b, make_float2(-8388736.0f, -8388736.0f));
}

// acc += sum over 8 elements of q_e * x_e (int8 codes w; x as fp32, elements
// 0..3 in xa and 4..7 in xb; every product is exact in fp32), as two
// partial sums (even, odd elements) with packed FMAs
__device__ __forceinline__ float2 dot8_q8x2(const uint2 w, const float4 xa, const float4 xb, float2 acc) {
    const uint32_t w0 = w.x ^ 0x80808080u, w1 = w.y ^ 0x80808080u;
    acc = __ffma2_rn(q8_pair(w0, 0), make_float2(xa.x, xa.y), acc);
    acc = __ffma2_rn(q8_pair(w0, 2), make_float2(xa.z, xa.w), acc);
    acc = __ffma2_rn(q8_pair(w1, 0), make_float2(xb.x, xb.y), acc);
    acc = __ffma2_rn(q8_pair(w1, 2), make_float2(xb.z, xb.w), acc);
    return acc;
}

// int4 weights: a word holds the offset-binary codes n = q + 8 of 8
// consecutive elements, element 2 j + h in bits 16 h + 4 j.  Masking nibble
// j of the low and of the high half-word and OR-ing in the exponent of 2^23
// gives the exact floats 2^23 + n 2^(4 j) (one LOP3 each); one packed FMA by
// 2^(-4 j) with addend -(2^(23 - 4 j) + 8) leaves q = n - 8 exactly (every
// intermediate value is an integer below 2^24).  The pair is elements
// (2 j, 2 j + 1), the two halves of bf16 word j of the same 8 elements.
template <int J>
__device__ __forceinline__ float2 q4_pair(uint32_t lo, uint32_t hi) {
    constexpr uint32_t m = 0xFu << (4 * J);
    constexpr float sc = 1.0f / (float)(1u << (4 * J));
    constexpr float off = -(float)(1u << (23 - 4 * J)) - 8.0f;
    const float2 b = make_float2(__uint_as_float((lo & m) | 0x4B000000u),
                                 __uint_as_float((hi & m) | 0x4B000000u));
    return __ffma2_rn(b, make_float2(sc, sc), make_float2(off, off));
}

// acc += sum over 8 elements of q_e * x_e (int4 codes w; x as in dot8_q8x2)
__device__ __forceinline__ float2 dot8_q4x2(const uint32_t w, const float4 xa, const float4 xb, float2 acc) {
    const uint32_t hi = w >> 16;
    acc = __ffma2_rn(q4_pair<0>(w, hi), make_float2(xa.x, xa.y), acc);
    acc = __ffma2_rn(q4_pair<1>(w, hi), make_float2(xa.z, xa.w), acc);
    acc = __ffma2_rn(q4_pair<2>(w, hi), make_float2(xb.x, xb.y), acc);
    acc = __ffma2_rn(q4_pair<3>(w, hi), make_float2(xb.z, xb.w), acc);
    return acc;
}

struct Stage2Args {
    const uint8_t* gateup;  // [F] rows of gu_row_bytes(d, WQ)
    const uint8_t* down_t;  // [F] rows of down_row_bytes(d, WQ)
    float* y;
    float* hch;     // [F] h per channel (debug, may be null)
    int* status;
    int d, F, n_gu, n_d, n_a;  // as in FusedParams
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

// Waits (every lane polls) until the shared-memory flag is set.  After two
// polls the warp sleeps between polls: a spinning warp takes issue slots
// from the warps on its scheduler that compute what it waits for (pass B
// waiting on pass A's h).
__device__ __forceinline__ bool warp_wait_flag(const uint8_t* flag, long long limit_ns, Ctl& ctl,
                                               int* status) {
    bool got = true;
    uint64_t t0 = 0;
    for (uint32_t it = 1; !*reinterpret_cast<const volatile uint8_t*>(flag); ++it) {
        if (it > 2) __nanosleep(32);
        if ((it & 63u) == 0) {
            if (*reinterpret_cast<volatile int*>(&ctl.abort)) {
                got = false;
                break;
            }
            const uint64_t now = global_timer_ns();
            if (t0 == 0) t0 = now;
            else if ((long long)(now - t0) > limit_ns) {
                got = false;
                ctl.abort = 1;
                record_status(status, PROX_ERR_TIMEOUT);
                break;
            }
        }
    }
    __threadfence_block();
    return __all_sync(0xffffffffu, got);
}

// Stage-2 roles of warps 0..17 over the CTA's items ctl.item[0..n), every
// item final when the roles start (the decode step resolves the exact mask
// first; the dense pass takes every channel of its chunk).
// Shared area: x as bf16 (2 d bytes), then n_gu gate|up stages, one row
// each (bf16 4 d bytes; int8: the codes 2 d + 16 bytes with the row's
// scales s_gate, s_up, s_down; int4 d + 16), then for bf16 n_d W_down^T
// stages of 2 d bytes, for codes the pass-B slots of n_d items
// (self_item_bytes each) and x once more as fp32 (4 d bytes).
//   GU producer (warp 16) / D producer (warp 17, bf16 only): the whole warp
//       issues, in rounds of W = min(32, stages) items (distinct stages):
//       lane j waits until the stage of item r W + j is free and issues its
//       bulk copy;
//   pass A (warp w < n_a, n_a dividing n_gu): the items i = w (mod n_a); item
//       i sits in gate|up stage i mod n_gu, whose items are all = w (mod
//       n_a), so one warp consumes each stage's uses in order (a parity wait
//       is never taken two uses ahead): g, u over the whole row,
//       h = silu(g) u, then ctl.hready[i] (codes: g and u times the row
//       scales, and ctl.h[i] = h s_down, the factor of the W_down^T codes);
//   pass B (warps 8..15): every thread owns 8-element slices of d and adds
//       h * W_down^T[c, slice] for the items in order; for bf16 rows from
//       the W_down^T ring, for codes from slots that each thread fills with
//       its own slices (see there).
// Stages and their phase parities advance by counters (no division).
template <int CPT, int WQ>
__device__ void stage2_roles(const Stage2Args& a, Ctl& ctl, uint8_t* area, int n) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d = a.d, n_gu = a.n_gu, n_d = a.n_d, n_a = a.n_a;
    const size_t gu_bytes = gu_row_bytes(d, WQ), d_bytes = down_row_bytes(d, WQ);
    const uint16_t* xs = reinterpret_cast<const uint16_t*>(area);
    uint8_t* gu_ring = area + (size_t)2 * d;
    uint8_t* d_ring = gu_ring + (size_t)n_gu * gu_bytes;
    const int nchunk = d / 8;  // 8-element chunks per row (16 bytes bf16, 8 int8, 4 int4)

    if (WQ != 0 && warp == kDProducerWarp) return;  // codes: pass B streams its own slices
    if (warp == kGuProducerWarp || warp == kDProducerWarp) {
        // The whole warp issues: in round r, lane j takes item r W + j
        // (W = min(32, stages), so a round's items use distinct stages),
        // waits until its stage is free and issues the bulk copy.
        const bool gu = warp == kGuProducerWarp;
        const int ns = gu ? n_gu : n_d;
        const int W = ns < 32 ? ns : 32;
        const size_t sb = gu ? gu_bytes : d_bytes;
        uint64_t* full = gu ? ctl.gu_full : ctl.d_full;
        uint64_t* empty = gu ? ctl.gu_empty : ctl.d_empty;
        int* last = gu ? ctl.gu_last : ctl.d_last;
        uint8_t* base = gu ? gu_ring : d_ring;
        const uint8_t* src = gu ? a.gateup : a.down_t;
        const uint64_t pol = policy_evict_first();
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (mbar_wait_bounded(bar, parity, a.limit_ns, &ctl.abort)) return true;
            if (!ctl.abort) {
                ctl.abort = 1;
                record_status(a.status, PROX_ERR_TIMEOUT);
            }
            return false;
        };
        for (int i0 = 0; i0 < n; i0 += W) {
            const int i = i0 + lane;
            bool ok = true;
            if (lane < W && i < n) {
                const int s = i % ns;
                if (i >= ns) ok = wait(&empty[s], ((i / ns) - 1) & 1);
                if (ok && !*reinterpret_cast<volatile int*>(&ctl.abort)) {
                    const int c = ctl.item[i];
                    if (c < 0 || c >= a.F) {  // never expected: the lists hold chunk channels
                        record_status(a.status, PROX_ERR_DEVICE_CHECK);
                        ctl.abort = 1;
                        ok = false;
                    } else {
                        last[s] = i;
                        mbar_arrive_expect_tx(&full[s], (uint32_t)sb);
                        bulk_g2s(base + (size_t)s * sb, src + (size_t)c * sb, (uint32_t)sb, &full[s], pol);
                    }
                }
            }
            if (!__all_sync(0xffffffffu, ok) || *reinterpret_cast<volatile int*>(&ctl.abort)) break;
        }
        return;
    }

    if (warp < kPassAWarps) {
        // ------------------------------------------------ pass A: h per item
        if (warp >= n_a) return;
        const uint4* xv = reinterpret_cast<const uint4*>(xs);
        // codes: the pass-A warps first write x as fp32 in two planes
        // (elements 0..3 and 4..7 of every 8-element chunk), so that a lane's
        // x loads are consecutive and no row converts x again
        float4* xfa = reinterpret_cast<float4*>(d_ring + (size_t)n_d * self_item_bytes(d, WQ));
        float4* xfb = xfa + nchunk;
        if constexpr (WQ != 0) {
            for (int ch = threadIdx.x; ch < nchunk; ch += n_a * 32) {
                const uint4 w = xv[ch];
                xfa[ch] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                                      __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
                xfb[ch] = make_float4(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u),
                                      __uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
            }
            named_barrier_sync(2, n_a * 32);  // warps 0 .. n_a - 1, each once
        }
        int s = warp;      // stage of item i
        uint32_t ph = 0;   // its phase parity
        for (int i = warp; i < n; i += n_a) {
            if (!warp_wait(&ctl.gu_full[s], ph, a.limit_ns, ctl, a.status)) break;
            if (i == 0 && lane == 0) stamp_here(a.ts, 6);
            const uint8_t* st = gu_ring + (size_t)s * gu_bytes;
            float g = 0.0f, u = 0.0f;
            if constexpr (WQ == 2) {
                const uint32_t* gr = reinterpret_cast<const uint32_t*>(st);
                const uint32_t* ur = gr + nchunk;
                float2 g2 = make_float2(0.0f, 0.0f), u2 = g2;
                for (int ch = lane; ch < nchunk; ch += 32) {
                    const float4 xa = xfa[ch], xb = xfb[ch];
                    g2 = dot8_q4x2(gr[ch], xa, xb, g2);
                    u2 = dot8_q4x2(ur[ch], xa, xb, u2);
                }
                g = g2.x + g2.y;
                u = u2.x + u2.y;
            } else if constexpr (WQ == 1) {
                const uint2* gr = reinterpret_cast<const uint2*>(st);
                const uint2* ur = gr + nchunk;
                float2 g2 = make_float2(0.0f, 0.0f), u2 = g2;
                for (int ch = lane; ch < nchunk; ch += 32) {
                    const float4 xa = xfa[ch], xb = xfb[ch];
                    g2 = dot8_q8x2(gr[ch], xa, xb, g2);
                    u2 = dot8_q8x2(ur[ch], xa, xb, u2);
                }
                g = g2.x + g2.y;
                u = u2.x + u2.y;
            } else {
                const uint4* gr = reinterpret_cast<const uint4*>(st);
                const uint4* ur = gr + nchunk;
                // bf16 -> fp32 is exact; two partial sums (even, odd
                // elements) with packed FMAs
                float2 g2 = make_float2(0.0f, 0.0f), u2 = g2;
                for (int ch = lane; ch < nchunk; ch += 32) {
                    const uint4 xw = xv[ch], gw = gr[ch], uw = ur[ch];
                    const uint32_t xa[4] = {xw.x, xw.y, xw.z, xw.w}, ga[4] = {gw.x, gw.y, gw.z, gw.w},
                                   ua[4] = {uw.x, uw.y, uw.z, uw.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 xf = make_float2(__uint_as_float(xa[e] << 16), __uint_as_float(xa[e] & 0xffff0000u));
                        g2 = __ffma2_rn(make_float2(__uint_as_float(ga[e] << 16), __uint_as_float(ga[e] & 0xffff0000u)), xf, g2);
                        u2 = __ffma2_rn(make_float2(__uint_as_float(ua[e] << 16), __uint_as_float(ua[e] & 0xffff0000u)), xf, u2);
                    }
                }
                g = g2.x + g2.y;
                u = u2.x + u2.y;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                g += __shfl_xor_sync(0xffffffffu, g, o);
                u += __shfl_xor_sync(0xffffffffu, u, o);
            }
            if (lane == 0) {
                float hs = 1.0f;  // factor of the W_down^T row
                if constexpr (WQ != 0) {  // the scales end the row
                    const float4 sc = *reinterpret_cast<const float4*>(st + gu_bytes - 16);
                    g *= sc.x;
                    u *= sc.y;
                    hs = sc.z;
                }
                mbar_arrive(&ctl.gu_empty[s]);
                const float h = g / (1.0f + expf(-g)) * u;  // silu(g) * u
                ctl.h[i] = WQ ? h * hs : h;
                if (a.hch) a.hch[ctl.item[i]] = h;
                __threadfence_block();
                *reinterpret_cast<volatile uint8_t*>(&ctl.hready[i]) = 1;
            }
            s += n_a;
            if (s >= n_gu) {
                s -= n_gu;
                ph ^= 1u;
            }
        }
        if (warp == 0 && lane == 0) stamp_here(a.ts, 7);
        return;
    }

    // ---------------------------------------------------- pass B: y += h W_down^T
    const int t = threadIdx.x - kPassBWarp0 * 32;
    float yp[CPT][8];
#pragma unroll
    for (int q = 0; q < CPT; ++q)
#pragma unroll
        for (int e = 0; e < 8; ++e) yp[q][e] = 0.0f;
    // y slice q += hv * the 8 weights of the chunk at p (q a constant
    // after unrolling)
    auto acc_chunk = [&](int q, const uint8_t* p, float hv) {
        const float2 h2 = make_float2(hv, hv);
        if constexpr (WQ == 2) {
            const uint32_t dw = *reinterpret_cast<const uint32_t*>(p);
            const uint32_t hi = dw >> 16;
            float2 a = __ffma2_rn(h2, q4_pair<0>(dw, hi), make_float2(yp[q][0], yp[q][1]));
            yp[q][0] = a.x;
            yp[q][1] = a.y;
            a = __ffma2_rn(h2, q4_pair<1>(dw, hi), make_float2(yp[q][2], yp[q][3]));
            yp[q][2] = a.x;
            yp[q][3] = a.y;
            a = __ffma2_rn(h2, q4_pair<2>(dw, hi), make_float2(yp[q][4], yp[q][5]));
            yp[q][4] = a.x;
            yp[q][5] = a.y;
            a = __ffma2_rn(h2, q4_pair<3>(dw, hi), make_float2(yp[q][6], yp[q][7]));
            yp[q][6] = a.x;
            yp[q][7] = a.y;
        } else if constexpr (WQ == 1) {
            const uint2 dw = *reinterpret_cast<const uint2*>(p);
            const uint32_t w0 = dw.x ^ 0x80808080u, w1 = dw.y ^ 0x80808080u;
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                float2 a = __ffma2_rn(h2, q8_pair(w0, e), make_float2(yp[q][e], yp[q][e + 1]));
                yp[q][e] = a.x;
                yp[q][e + 1] = a.y;
                a = __ffma2_rn(h2, q8_pair(w1, e), make_float2(yp[q][4 + e], yp[q][5 + e]));
                yp[q][4 + e] = a.x;
                yp[q][5 + e] = a.y;
            }
        } else {
            const uint4 dw = *reinterpret_cast<const uint4*>(p);
            const uint32_t dv[4] = {dw.x, dw.y, dw.z, dw.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 a = __ffma2_rn(h2, make_float2(__uint_as_float(dv[e] << 16), __uint_as_float(dv[e] & 0xffff0000u)),
                                            make_float2(yp[q][2 * e], yp[q][2 * e + 1]));
                yp[q][2 * e] = a.x;
                yp[q][2 * e + 1] = a.y;
            }
        }
    };
    constexpr size_t chunk_bytes = WQ == 2 ? 4 : WQ == 1 ? 8 : 16;
    auto add_row = [&](const uint8_t* row, float hv) {
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
            const int ch = t + q * kPassB;
            if (ch < nchunk) acc_chunk(q, row + (size_t)ch * chunk_bytes, hv);
        }
    };
    bool ok = true;
    if constexpr (WQ != 0) {
        // Codes: thread t copies its own chunks of each item's W_down^T row
        // (cp.async of 8 or 4 bytes) n_d items ahead into its slots and
        // waits only for its own copies (one cp.async group per item), so
        // no stage barriers and no producer warp are involved.  Slot (k, q)
        // of thread t: d_ring + ((k CPT + q) kPassB + t) cb bytes.
        constexpr int cb = WQ == 2 ? 4 : 8;
        const int K = n_d;  // 2, 4 or 8
        const uint64_t pol = policy_evict_first();
        auto slot = [&](int k, int q) { return d_ring + ((size_t)(k * CPT + q) * kPassB + t) * cb; };
        auto issue = [&](int i, int k) {
            const uint8_t* row = a.down_t + (size_t)ctl.item[i] * d_bytes;
#pragma unroll
            for (int q = 0; q < CPT; ++q) {
                const int ch = t + q * kPassB;
                if (ch < nchunk) cp_async_small<cb>(slot(k, q), row + (size_t)ch * cb, pol);
            }
        };
        for (int j = 0; j < K; ++j) {
            if (j < n) issue(j, j);
            cp_async_commit();
        }
        int k = 0;
        for (int i = 0; i < n; ++i) {
            if (K == 8) cp_async_wait_group<7>();  // item i's group has landed
            else if (K == 4) cp_async_wait_group<3>();
            else cp_async_wait_group<1>();
            ok = warp_wait_flag(&ctl.hready[i], a.limit_ns, ctl, a.status);
            if (!ok) break;
            const float hv = *reinterpret_cast<const volatile float*>(&ctl.h[i]);
#pragma unroll
            for (int q = 0; q < CPT; ++q)
                if (t + q * kPassB < nchunk) acc_chunk(q, slot(k, q), hv);
            if (i + K < n) issue(i + K, k);  // into the slot just read
            cp_async_commit();
            if (++k == K) k = 0;
        }
        cp_async_wait_group<0>();  // nothing in flight when the CTA leaves
    } else {
        // bf16: the W_down^T ring, one item per step (two per step, waiting
        // for two of its 6 stages, measured slower)
        int s = 0;         // stage of item i
        uint32_t ph = 0;   // its phase parity
        for (int i = 0; i < n; ++i) {
            ok = warp_wait(&ctl.d_full[s], ph, a.limit_ns, ctl, a.status) &&
                 warp_wait_flag(&ctl.hready[i], a.limit_ns, ctl, a.status);
            if (!ok) break;
            add_row(d_ring + (size_t)s * d_bytes, *reinterpret_cast<const volatile float*>(&ctl.h[i]));
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.d_empty[s]);
            if (++s == n_d) {
                s = 0;
                ph ^= 1u;
            }
        }
    }
    if (t == 0) stamp_here(a.ts, 8);
    if (ok && !ctl.abort && n > 0) {
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
            const int ch = t + q * kPassB;
            if (ch < nchunk) {
                float* dst = a.y + (size_t)ch * 8;
                red_add_v4(dst, yp[q][0], yp[q][1], yp[q][2], yp[q][3]);
                red_add_v4(dst + 4, yp[q][4], yp[q][5], yp[q][6], yp[q][7]);
            }
        }
    }
}

// Initialises the Stage-2 ring barriers (one thread; the caller
// synchronises).  reinit: an earlier step of this launch initialised them
// (same ring geometry), so they are invalidated first.
__device__ __forceinline__ void stage2_init(Ctl& ctl, int n_gu, int n_d, bool reinit = false) {
    if (reinit) {
        for (int s = 0; s < n_gu; ++s) {
            mbar_inval(&ctl.gu_full[s]);
            mbar_inval(&ctl.gu_empty[s]);
        }
        for (int s = 0; s < n_d; ++s) {
            mbar_inval(&ctl.d_full[s]);
            mbar_inval(&ctl.d_empty[s]);
        }
        mbar_inval(&ctl.done_bar);
    }
    for (int s = 0; s < n_gu; ++s) {
        mbar_init(&ctl.gu_full[s], 1);
        mbar_init(&ctl.gu_empty[s], 1);
        ctl.gu_last[s] = -1;
    }
    for (int s = 0; s < n_d; ++s) {
        mbar_init(&ctl.d_full[s], 1);
        mbar_init(&ctl.d_empty[s], kPassBWarps);
        ctl.d_last[s] = -1;
    }
    mbar_init(&ctl.done_bar, kNT / 32);
}

// End of the Stage-2 roles: every warp, once its lanes are through, arrives
// on ctl.done_bar; thread 0 waits for all of them (the roles are warp-
// specialised, so a block barrier is not used here), stamps the end and,
// after an abort, lets the bulk copies still in flight into the rings land
// before the CTA leaves (bounded).  Pass-B threads that stream code slices
// wait for their own cp.async copies before they arrive.
__device__ __forceinline__ void stage2_join(const Stage2Args& a, Ctl& ctl) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&ctl.done_bar);
    if (threadIdx.x != 0) return;
    mbar_wait_bounded(&ctl.done_bar, 0, a.limit_ns, nullptr);
    stamp_here(a.ts, 9);
    if (!ctl.abort) return;
    for (int s = 0; s < a.n_gu; ++s)
        if (ctl.gu_last[s] >= 0)
            mbar_wait_bounded(&ctl.gu_full[s], (ctl.gu_last[s] / a.n_gu) & 1, a.limit_ns, nullptr);
    for (int s = 0; s < a.n_d; ++s)
        if (ctl.d_last[s] >= 0)
            mbar_wait_bounded(&ctl.d_full[s], (ctl.d_last[s] / a.n_d) & 1, a.limit_ns, nullptr);
}

// ------------------------------------------------------------ the selection
// Certain rows per CTA prefetched into L2 during the selection.  Each bulk
// prefetch costs issue time in the selection's path: 8 rows (~28 MB over the
// grid) measured best; 16, 24 and 32 delayed the mask by up to 1.6 us.
constexpr int kPrefetchItems = 8;

// Bulk prefetch of global memory into L2 (no shared-memory destination).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}


// Block-wide digit select, called by every thread: threads t < NB/4 read
// bins 4t..4t+3 with one 16-byte load (consecutive threads, consecutive
// words: no bank conflict) and a suffix sum from the top bin finds the bin b
// with sum(h[b+1..]) < krem <= sum(h[b..]); (b, krem - sum(h[b+1..])) go to
// ctl.sel[0..1].  If the bins hold fewer than krem counts ctl.sel[0] stays
// 0xffffffff.
template <int NB>
__device__ __forceinline__ void block_select(const uint32_t* h, uint32_t krem, Ctl& ctl,
                                             const uint32_t* hg = nullptr) {
    constexpr int NQ = NB / 4, NW = NQ / 32;
    static_assert(NQ % 32 == 0 && NQ <= kNT, "bins");
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    // the bins from shared memory, or (hg given) from global memory through L2
    if (tid < NQ) v = hg ? __ldcg(reinterpret_cast<const uint4*>(hg) + tid)
                         : reinterpret_cast<const uint4*>(h)[tid];
    const uint32_t s = (v.x + v.y) + (v.z + v.w);
    uint32_t suf = s;  // sum over this and the higher lanes of the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += t;
    }
    if (wid < NW && lane == 0) ctl.warp_tot[wid] = suf;
    if (tid == 0) ctl.sel[0] = 0xffffffffu;
    __syncthreads();
    if (tid < NQ) {
        uint32_t above = suf - s;
        if constexpr (NW > 1) {  // the higher warps' totals: independent 16-byte loads
            constexpr int NV = (NW + 3) / 4;
            uint4 wt[NV];
#pragma unroll
            for (int q = 0; q < NV; ++q) wt[q] = reinterpret_cast<const uint4*>(ctl.warp_tot)[q];
#pragma unroll
            for (int q = 0; q < NV; ++q) {
                const uint32_t x4[4] = {wt[q].x, wt[q].y, wt[q].z, wt[q].w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (4 * q + e < NW && 4 * q + e > wid) above += x4[e];
            }
        }
        if (above < krem && above + s >= krem) {
            // the bin within this thread's four, top bin first (no indexed array)
            uint32_t j = 3, a = above;
            if (a + v.w < krem) {
                a += v.w;
                j = 2;
                if (a + v.z < krem) {
                    a += v.z;
                    j = 1;
                    if (a + v.y < krem) {
                        a += v.y;
                        j = 0;
                    }
                }
            }
            ctl.sel[0] = 4u * (uint32_t)tid + j;
            ctl.sel[1] = krem - a;
        }
    }
    __syncthreads();
}

// Every CTA, all threads, once every channel's score key is published
// (grid barrier 2): the exact channel top-k and this CTA's share of it.
// HBM is idle at this point, so the reads below are L2 hits at low latency:
// the digit-1 histogram (every chunk added to it) straight into the threads
// that select on it, and all F score keys (channel order) into shared
// memory by one bulk copy, which lands while digit 1 is being selected.
//   digit 1 (bits 30..20 of the score bits) of the k-th key from the
//   global histogram; digit 2 (bits 19..9) and digit 3 (bits 8..0) from
//   shared histograms over the keys in the digit-1 bin (the candidates);
//   then T (the k-th key) and r (keys equal to T to keep, lowest channels
//   first).  Thread t owns the keys [t kpt, (t+1) kpt); one block scan of
//   (keys above T, keys equal to T) per thread gives each thread the
//   position of its first selected channel in the ascending list of
//   selected channels; CTA b takes the positions [k b / n, k (b+1) / n) of
//   that list as its Stage-2 items (an even split: every CTA moves the same
//   bytes; every CTA computes the same T and prefixes, so the shares
//   partition the mask).
// Costs measured on this part drove the layout: a block-wide select or scan
// costs ~1000 cycles, a pass over all keys ~1500, and a shared store or
// atomic inside a loop that loads from shared memory serialises each step,
// so every pass over keys is loads-only and builds bit masks.  While it
// runs, the first certain rows of the CTA's own chunk stream into L2.
// Returns false on a timeout or a broken invariant (ctl.abort set).
__device__ bool select_items(const FusedParams& p, Ctl& ctl, uint8_t* area, int nb, int b,
                             int cb0, int nch) {
    const int tid = threadIdx.x;
    // the ranked keys: one per channel, or one per block of bw channels (a
    // block mask: its K = k / bw largest blocks, every channel of each)
    const int bw = p.bw > 0 ? p.bw : 1;
    const int F = p.F / bw, kk_sel = p.k / bw;
    const uint32_t kbytes = (uint32_t)((F * 4 + 15) / 16 * 16);
    uint32_t* h2 = reinterpret_cast<uint32_t*>(area + (size_t)2 * p.d);
    uint32_t* h3 = h2 + kHistBins;
    uint32_t* sk = h3 + 512;  // [F] score keys, channel (block) order
    if (tid == 0) {
        asm volatile("fence.proxy.async.global;" ::: "memory");
        const uint64_t pol = policy_evict_first();
        mbar_arrive_expect_tx(&ctl.key_ld, kbytes);
        bulk_g2s(sk, p.skey, kbytes, &ctl.key_ld, pol);
    }
    for (int i = tid; i < kHistBins + 512; i += kNT) h2[i] = 0u;
    // waits for one of the staging copies; after a timeout lets both land
    // (one thread polls the barrier; the block barrier then orders the data
    // for every thread: 608 threads polling one mbarrier cost ~600 cycles)
    auto landed = [&](uint64_t* bar) {
        if (tid == 0 && !mbar_wait_bounded(bar, 0, p.limit_ns, &ctl.abort)) {
            ctl.abort = 1;
            record_status(p.status, PROX_ERR_TIMEOUT);
        }
        __syncthreads();
        if (!ctl.abort) return true;
        if (tid == 0) {
            mbar_wait_bounded(&ctl.key_ld, 0, p.limit_ns, nullptr);
        }
        return false;
    };
    auto broken = [&]() {
        if (tid == 0) {
            record_status(p.status, PROX_ERR_DEVICE_CHECK);
            ctl.abort = 1;
            mbar_wait_bounded(&ctl.key_ld, 0, p.limit_ns, nullptr);  // before the area is reused
        }
        __syncthreads();
        return false;
    };
    // digit 1 from the histogram of every chunk, read from L2 straight into
    // the selecting threads (the keys still landing)
    block_select<2048>(nullptr, (uint32_t)kk_sel, ctl, p.hist);
    stamp(p.ts, 14);
    if (ctl.sel[0] == 0xffffffffu) return broken();
    const uint32_t b1 = ctl.sel[0], k1 = ctl.sel[1];
    // own channels above the digit-1 bin are certain members of the mask:
    // rank them in channel order (the barrier inside landed publishes the
    // warp counts); once the keys are in (no more staging traffic to delay),
    // the first kPrefetchItems of them start streaming into L2, each by its
    // own thread, while the rest of the selection runs; the CTA whose share
    // holds them finds them in L2 (shares follow channel order, so mostly
    // this CTA or a neighbour)
    const bool sure = tid < min(nch, kMaxChunk) && (__float_as_uint(ctl.lsc[tid]) >> 20) > b1;
    const unsigned sb = __ballot_sync(0xffffffffu, sure);
    if ((tid & 31) == 0) ctl.warp_tot[tid >> 5] = __popc(sb);
    if (!landed(&ctl.key_ld)) return false;
    if (sure) {
        int rank = __popc(sb & ((1u << (tid & 31)) - 1u));
        for (int w = 0; w < (tid >> 5); ++w) rank += (int)ctl.warp_tot[w];  // nch <= 256: <= 7 warps
        if (rank < kPrefetchItems && !p.member) {  // mask only: the rows are read later
            const int c = cb0 + tid;
            const size_t gb = gu_row_bytes(p.d, p.wq), db = down_row_bytes(p.d, p.wq);
            prefetch_l2(p.gateup + (size_t)c * gb, (uint32_t)gb);
            prefetch_l2(p.down_t + (size_t)c * db, (uint32_t)db);
        }
    }
    // Thread t owns the keys [i0, i1) = [t kpt, (t+1) kpt) (channel order).
    // kpt is odd, so the threads of a warp stepping through their keys
    // together hit 32 different shared-memory banks (an even stride such as
    // 24 puts 8 of them on each bank).  Every loop over keys is loads-only:
    // on this part a shared store or atomic inside a loop that also loads
    // from shared memory serialises each step (~200 cycles instead of ~20),
    // so the passes build per-thread bit masks (kpt <= 55 < 64) and the
    // stores come afterwards, over the few set bits.
    const int kpt = ((F + kNT - 1) / kNT) | 1;
    const int i0 = min(F, tid * kpt), n = min(F, i0 + kpt) - i0;
    const uint32_t* mk = sk + i0;
    uint64_t above = 0, cmask = 0;  // keys above the digit-1 bin / in it (candidates)
    for (int e = 0; e < n; ++e) {
        const uint32_t d1 = mk[e] >> 20;
        above |= (uint64_t)(d1 > b1) << e;
        cmask |= (uint64_t)(d1 == b1) << e;
    }
    for (uint64_t m = cmask; m; m &= m - 1) {
        const uint32_t kk = mk[__ffsll((long long)m) - 1];
        atomicAdd(&h2[(kk >> 9) & 2047u], 1u);
    }
    __syncthreads();
    block_select<2048>(h2, k1, ctl);
    if (ctl.sel[0] == 0xffffffffu) return broken();
    const uint32_t pre = (b1 << 11) | ctl.sel[0], k2 = ctl.sel[1];
    // digit 3 over the candidates matching both digits
    for (uint64_t m = cmask; m; m &= m - 1) {
        const uint32_t kk = mk[__ffsll((long long)m) - 1];
        if ((kk >> 9) == pre) atomicAdd(&h3[kk & 511u], 1u);
    }
    __syncthreads();
    block_select<512>(h3, k2, ctl);
    if (ctl.sel[0] == 0xffffffffu) return broken();
    const uint32_t T = (pre << 9) | ctl.sel[0];
    const uint32_t r = ctl.sel[1];  // keys equal to T to keep, lowest channels first
    stamp(p.ts, 15);
    // this thread's keys above T and equal to T (T lies in the digit-1 bin,
    // so only the candidates need a look); one scan gives the selected
    // channels and the ties before this thread (counts <= F <= 32768 < 2^16)
    uint64_t gtm = above, eqm = 0;
    for (uint64_t m = cmask; m; m &= m - 1) {
        const int e = __ffsll((long long)m) - 1;
        const uint32_t kk = mk[e];
        if (kk > T) gtm |= 1ull << e;
        else if (kk == T) eqm |= 1ull << e;
    }
    const uint32_t gt = (uint32_t)__popcll(gtm), eq = (uint32_t)__popcll(eqm);
    uint32_t tot;
    const uint32_t ex = block_excl_scan<kNT>(gt | (eq << 16), ctl, tot);
    const uint32_t ties = ex >> 16;
    const uint32_t pos = (ex & 0xffffu) + min(ties, r);  // selected channels before this thread's
    if ((tot & 0xffffu) + min(tot >> 16, r) != (uint32_t)kk_sel) return broken();
    const int q0 = chunk_begin(p.k, b, nb), q1 = chunk_begin(p.k, b + 1, nb);
    if (q1 - q0 > kMaxItems) return broken();
    // the ties this thread keeps: its lowest min(eq, r - ties) tie bits
    uint32_t keep = ties < r ? min(eq, r - ties) : 0u;
    uint64_t sel = gtm;
    for (uint64_t m = eqm; m && keep; m &= m - 1, --keep) sel |= m & (~m + 1);
    // a thread whose selected keys meet the channel positions [q0, q1) writes
    // those items (a selected block at position j holds the channel
    // positions [j bw, (j + 1) bw)); in debug mode CTA 0 writes the whole mask
    const int nsel = __popcll(sel);
    if ((int)pos * bw < q1 && ((int)pos + nsel) * bw > q0) {
        int at = (int)pos * bw;
        for (uint64_t m = sel; m && at < q1; m &= m - 1) {
            const int c = (i0 + __ffsll((long long)m) - 1) * bw;
            for (int j = 0; j < bw; ++j, ++at)
                if (at >= q0 && at < q1) ctl.item[at - q0] = c + j;
        }
    }
    if (p.debug && b == 0) {
        int at = (int)pos * bw;
        for (uint64_t m = sel; m; m &= m - 1) {
            const int c = (i0 + __ffsll((long long)m) - 1) * bw;
            for (int j = 0; j < bw; ++j, ++at) p.idx_list[at] = c + j;
        }
    }
    if (tid == 0) ctl.n_items = q1 - q0;
    __syncthreads();
    return true;
}

// ------------------------------------------------------------ fused kernel
// One decode step (one layer) inside a persistent launch.  The grid
// barrier word counts arrivals and is never reset between launches: gen is
// the number of grid barriers completed before this launch (read at its
// start), and this step's two barriers are number gen + bi + 1 and
// gen + bi + 2 (barrier j completes when the word reaches n j); bi > 0
// marks a later step of a stacked launch (its mbarriers are re-used).  The last
// step of a launch publishes gen + bi + 2 for the next launch (every CTA
// has read gen by then).  Returns false when the CTA must leave (a wait ran
// out or a check failed; the status word says which).
// GROUPED: the grid is split into groups of p.gsize CTAs (k_prox_masks);
// a group's CTA chunks can then be wider than the CTA's threads.
template <int CPT, int WQ, bool GROUPED = false>
__device__ __forceinline__ bool fused_step(const FusedParams& p, Ctl& ctl, uint8_t* area,
                                           unsigned gen, unsigned bi, bool last) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    // the CTAs that share this step: the whole grid, or this CTA's group
    const int nb = GROUPED ? p.gsize : (int)gridDim.x;
    const int b = GROUPED ? (int)blockIdx.x % p.gsize : (int)blockIdx.x;
    const int d = p.d, F = p.F, Fp = p.Fp;
    stamp(p.ts, 0);
    // a later step of a stacked launch finds the barriers of the step before
    // it still valid in shared memory: invalidate, then initialise
    const bool reinit = bi > 0;
    if (tid == 0) {
        if (reinit) mbar_inval(&ctl.ld_bar);
        mbar_init(&ctl.ld_bar, 1);
        fence_mbar_init();
    } else if (tid == kNT - 32) {
        // the barriers of the selection and of Stage 2 (this warp has no x
        // group at the common sizes, so the set-up costs the input phase nothing)
        stage2_init(ctl, p.n_gu, p.n_d, reinit);
        if (reinit) mbar_inval(&ctl.key_ld);
        mbar_init(&ctl.key_ld, 1);
        fence_mbar_init();
    }
    for (int i = tid; i < kMaxItems; i += kNT) ctl.hready[i] = 0;

    // ------------------------------------------------ P0: input sparsity
    // area: x bf16 [d] | kept u32 [d] | histograms u32 [256 + 128] | P1 tables
    // Thread t holds the x groups [t G, (t+1) G) (8 bf16 each) in registers,
    // so the passes over the 15-bit keys |x| touch no memory; exact top-k_x in
    // two radix digits: the exponent (bits 14..7) and the 7 mantissa bits.
    uint16_t* xs = reinterpret_cast<uint16_t*>(area);
    uint32_t* kept = reinterpret_cast<uint32_t*>(area + (size_t)2 * d);
    uint32_t* hA = kept + d;
    uint32_t* hB = hA + 256;
    {
        const int ng = d / 8, G = (ng + kNT - 1) / kNT, g0 = tid * G;  // G <= kXGroups
        uint4 xv[kXGroups];
        auto valid = [&](int q) { return q < G && g0 + q < ng; };
        if (p.x_prev == nullptr) {
#pragma unroll
            for (int q = 0; q < kXGroups; ++q)
                xv[q] = valid(q) ? __ldg(reinterpret_cast<const uint4*>(p.x) + g0 + q)
                                 : make_uint4(0u, 0u, 0u, 0u);
        } else {
            // stack glue: z = x_prev + y_prev, x = bf16_rne(z / sqrt(mean(z^2) + eps)).
            // Every CTA sums z^2 in the same fixed order (thread-local, warp
            // butterfly, then the warps in order), so all CTAs get the same x.
            float z[kXGroups][8];
            float ss = 0.0f;
#pragma unroll
            for (int q = 0; q < kXGroups; ++q) {
                uint4 xb = make_uint4(0u, 0u, 0u, 0u);
                float4 y0 = make_float4(0.f, 0.f, 0.f, 0.f), y1 = y0;
                if (valid(q)) {
                    // through L2: a stacked launch wrote them in an earlier layer
                    xb = __ldcg(reinterpret_cast<const uint4*>(p.x_prev) + g0 + q);
                    y0 = __ldcg(reinterpret_cast<const float4*>(p.y_prev) + 2 * (g0 + q));
                    y1 = __ldcg(reinterpret_cast<const float4*>(p.y_prev) + 2 * (g0 + q) + 1);
                }
                const uint32_t w[4] = {xb.x, xb.y, xb.z, xb.w};
                const float yy[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t hb = (e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xffffu);
                    z[q][e] = __uint_as_float(hb << 16) + yy[e];
                    ss = fmaf(z[q][e], z[q][e], ss);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (lane == 0) ctl.warp_tot[wid] = __float_as_uint(ss);
            __syncthreads();
            float tot = 0.0f;
#pragma unroll
            for (int w = 0; w < kNT / 32; ++w) tot += __uint_as_float(ctl.warp_tot[w]);
            const float inv = 1.0f / sqrtf(tot / (float)d + p.eps);
#pragma unroll
            for (int q = 0; q < kXGroups; ++q) {
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    o[e] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(z[q][2 * e] * inv)) |
                           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(z[q][2 * e + 1] * inv)) << 16);
                xv[q] = make_uint4(o[0], o[1], o[2], o[3]);
                if (valid(q) && b == 0 && p.x_out)
                    reinterpret_cast<uint4*>(p.x_out)[g0 + q] = xv[q];
            }
            __syncthreads();  // ctl.warp_tot is reused below
        }
        auto half = [&](const uint4& v, int e) {
            const uint32_t w = e < 2 ? v.x : e < 4 ? v.y : e < 6 ? v.z : v.w;
            return (e & 1) ? (w >> 16) : (w & 0xffffu);
        };
        for (int i = tid; i < 384; i += kNT) hA[i] = 0u;
        if (tid == 0) ctl.sel[3] = 0u;
        if (b == 0) {
            for (int i = tid; i < d; i += kNT) p.y[i] = 0.0f;
            for (int i = tid; i < kHistWords; i += kNT) p.hist[i] = 0u;
        }
        __syncthreads();
        uint32_t mk = 0;
#pragma unroll
        for (int q = 0; q < kXGroups; ++q)
            if (valid(q)) {
                reinterpret_cast<uint4*>(xs)[g0 + q] = xv[q];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t kk = half(xv[q], e) & 0x7fffu;
                    mk = max(mk, kk);
                    atomicAdd(&hA[kk >> 7], 1u);
                }
            }
        mk = __reduce_max_sync(0xffffffffu, mk);
        if (lane == 0) atomicMax(&ctl.sel[3], mk);
        __syncthreads();
        stamp(p.ts, 10);
        if (tid == 0) {  // power-of-two prescale: max|x| * 2^shift in [2^14, 2^15)
            const uint32_t mx = ctl.sel[3];
            int sh = 0;
            if (mx != 0) {
                int ex;
                frexpf(__uint_as_float(mx << 16), &ex);  // max|x| in [2^(ex-1), 2^ex)
                sh = 15 - ex;
            }
            ctl.sel[2] = (uint32_t)sh;
        }
        block_select<256>(hA, (uint32_t)p.kx, ctl);
        const uint32_t b1 = ctl.sel[0], k1 = ctl.sel[1];
#pragma unroll
        for (int q = 0; q < kXGroups; ++q)
            if (valid(q))
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t kk = half(xv[q], e) & 0x7fffu;
                    if ((kk >> 7) == b1) atomicAdd(&hB[kk & 127u], 1u);
                }
        __syncthreads();
        block_select<128>(hB, k1, ctl);
        const uint32_t T = (b1 << 7) | ctl.sel[0], r = ctl.sel[1];
        uint32_t gt = 0, eq = 0;
#pragma unroll
        for (int q = 0; q < kXGroups; ++q)
            if (valid(q))
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t kk = half(xv[q], e) & 0x7fffu;
                    gt += kk > T;
                    eq += kk == T;
                }
        uint32_t tot;
        const uint32_t ex = block_excl_scan<kNT>(gt | (eq << 16), ctl, tot);
        uint32_t tie = ex >> 16;
        uint32_t pos = (ex & 0xffffu) + min(tie, r);  // kept entries before this thread's
        const int shift = (int)ctl.sel[2];
#pragma unroll
        for (int q = 0; q < kXGroups; ++q)
            if (valid(q))
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t hb = half(xv[q], e), kk = hb & 0x7fffu;
                    bool keep = kk > T;
                    if (kk == T) keep = tie++ < r;
                    if (keep) {
                        const int j = (g0 + q) * 8 + e;
                        kept[pos] = ((uint32_t)j << 16) | scaled_fp16((uint16_t)hb, shift);
                        if (b == 0 && p.kept_out) p.kept_out[pos] = j;
                        ++pos;
                    }
                }
    }
    __syncthreads();
    const int shift = (int)ctl.sel[2];
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
        const int r0 = chunk_begin(p.kx, slice, p.slices);  // kx <= 16384, slices <= 16
        const int r1 = chunk_begin(p.kx, slice + 1, p.slices);
        // row-lane rl takes the contiguous kept rows [q_beg, q_end)
        const int m = (r1 - r0 + R - 1) / R;
        const int q_beg = min(r1, r0 + rl * m), q_end = min(r1, q_beg + m);
        // per-thread ring of proxy row segments in flight, [kRing][kNT]; after
        // the rows are in, the running totals [R][16][tpr] float2 (channel
        // cu * 16 + t of row-lane rl at (rl * 16 + t) * tpr + cu, so a warp's
        // lanes touch consecutive 8-byte words) take its place
        uint4* ring = reinterpret_cast<uint4*>(hA + 1024);
        float2* tot = reinterpret_cast<float2*>(ring);
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
            mbar_arrive_expect_tx(&ctl.ld_bar, (uint32_t)(ng * width * 4));
            for (int g = 0; g < ng; ++g)
                bulk_g2s(ssc + (size_t)g * W, p.scales + (size_t)(g_lo + g) * Fp + c0,
                         (uint32_t)(width * 4), &ctl.ld_bar, pol);
        }
        // this group's sums (ag, au: sum n x in units of 2^-24 / 2^-20), the
        // group's sum of x (cx) and the scaled running totals (tg, tu)
        float ag[16], au[16], tg[16], tu[16];
        float cx = 0.0f;
#pragma unroll
        for (int t = 0; t < 16; ++t) ag[t] = au[t] = tg[t] = tu[t] = 0.0f;
        int cur_g = -1;
        bool scales_in = false;
        auto flush = [&]() {
            if (cur_g < 0) return;
            const uint4* src;
            if (smem_scales) {
                if (!scales_in) {
                    if (!mbar_wait_bounded(&ctl.ld_bar, 0, p.limit_ns, &ctl.abort)) {
                        ctl.abort = 1;
                        record_status(p.status, PROX_ERR_TIMEOUT);
                    }
                    scales_in = true;
                }
                src = reinterpret_cast<const uint4*>(ssc + (size_t)(cur_g - g_lo) * W + cu * 16);
            } else {
                src = reinterpret_cast<const uint4*>(p.scales + (size_t)cur_g * Fp + c0 + cu * 16);
            }
            const float m8c = -8.0f * cx;  // the offset: sum q x = sum n x - 8 sum x
            cx = 0.0f;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 s4 = src[v];
                const uint32_t sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = 4 * v + e;
                    const float2 s2 = __half22float2(*reinterpret_cast<const __half2*>(&sv[e]));
                    tg[t] = fmaf(s2.x, fmaf(ag[t], 16777216.0f, m8c), tg[t]);
                    tu[t] = fmaf(s2.y, fmaf(au[t], 1048576.0f, m8c), tu[t]);
                    ag[t] = 0.0f;
                    au[t] = 0.0f;
                }
            }
        };
        if (active && q_beg < q_end) {
            // kRing rows in flight per thread through a cp.async ring in
            // shared memory (slot s of thread t at ring[s * kNT + t]); each
            // thread reads only its own slots, so no block synchronisation.
            // With tpr a multiple of 16 (the whole-grid step) the row, and
            // kept[q], is uniform across each half-warp; other widths (group
            // launches) only split some warps over two rows.  One row per
            // iteration keeps the loop body (and its instruction footprint)
            // small.
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
                if (q == q_beg) stamp(p.ts, 11);
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
                fma_f32_f16(cx, (uint16_t)0x3C00u, xh);
                proxy_mac_word(w.x, xh, &ag[0], &au[0]);
                proxy_mac_word(w.y, xh, &ag[4], &au[4]);
                proxy_mac_word(w.z, xh, &ag[8], &au[8]);
                proxy_mac_word(w.w, xh, &ag[12], &au[12]);
            }
            cp_async_wait_group<0>();
            flush();
            stamp(p.ts, 12);
        }
        // the scale copy must have landed before this shared memory is reused
        if (smem_scales && !scales_in)
            if (!mbar_wait_bounded(&ctl.ld_bar, 0, p.limit_ns, &ctl.abort)) {
                ctl.abort = 1;
                record_status(p.status, PROX_ERR_TIMEOUT);
            }
        __syncthreads();  // every thread is done with its ring slots
        if (active)
#pragma unroll
            for (int t = 0; t < 16; ++t)
                tot[((size_t)rl * 16 + t) * tpr + cu] = make_float2(tg[t], tu[t]);
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
    if (!grid_barrier(p.bar, (unsigned)nb * (gen + bi + 1u), p.status, p.limit_ns, ctl,
                      p.inject == 1 && b == nb - 1))
        return false;
    stamp(p.ts, 3);

    // ------------------------------------------------ P2: scores + histogram
    const int cb0 = chunk_lo(F, b, nb, chunk_align(p.bw));
    const int cb1 = chunk_lo(F, b + 1, nb, chunk_align(p.bw));
    const int nch = cb1 - cb0;  // <= kMaxChunk, except in a group launch (block masks: always)
    // a group launch's chunk can be wider than the CTA: pieces of kNT channels
    // (the per-chunk scores in ctl.lsc cover the first kMaxChunk; they serve
    // the block mask and the L2 prefetch, neither of which a group launch uses)
    const int npieces = GROUPED ? (nch + kNT - 1) / kNT : 1;
    for (int piece = 0; piece < npieces; ++piece) {
        const int ci = piece * kNT + tid;
        const bool act = ci < nch;
        uint32_t key = 0;
        if (act) {
            const int c = cb0 + ci;
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
            // |silu(g~) * u~|, silu(z) = z / (1 + e^-z); the contribution
            // signal weights it by the norm of the W_down column it scales
            float sc = fabsf(g / (1.0f + expf(-g)) * u);
            if (p.dnorm) sc *= __ldg(p.dnorm + c);
            if (p.scores_out) p.scores_out[c] = sc;
            if (ci < kMaxChunk) ctl.lsc[ci] = sc;
            key = __float_as_uint(sc);
        }
        if (p.bw > 0) {
            // block-granular mask: every channel takes the sum of its block's
            // scores (blocks are bw consecutive threads, bw | chunk start).
            // Fixed order: a butterfly over min(bw, 32) lanes (every lane of a
            // group ends with the same sum), then the warp sums of a wider
            // block added in warp order.
            const int bw = p.bw;
            float sblk = act ? __uint_as_float(key) : 0.0f;
            for (int o = 1; o < bw && o < 32; o <<= 1) sblk += __shfl_xor_sync(0xffffffffu, sblk, o);
            if (bw > 32) {
                if (lane == 0) ctl.warp_tot[wid] = __float_as_uint(sblk);
                __syncthreads();
                if (act) {  // tid < nch <= kMaxChunk: warps 0 .. kMaxChunk / 32 - 1
                    const int w0 = (tid - tid % bw) >> 5;
                    float t = 0.0f;
                    for (int w = 0; w < (bw >> 5); ++w) t += __uint_as_float(ctl.warp_tot[w0 + w]);
                    sblk = t;
                }
                __syncthreads();  // ctl.warp_tot is reused below
            }
            if (act) {
                key = __float_as_uint(sblk);
                ctl.lsc[tid] = sblk;
            }
        }
        // the key, in channel order, for the selection; one histogram
        // reduction per distinct bin in the warp.  A block mask ranks blocks:
        // one key and one count per block, from its first channel (chunks
        // start on block boundaries)
        const bool pub = act && (p.bw == 0 || ((cb0 + ci) & (p.bw - 1)) == 0);
        if (pub) p.skey[p.bw ? (cb0 + ci) / p.bw : cb0 + ci] = key;
        const unsigned am = __ballot_sync(0xffffffffu, pub);
        if (pub) {
            const unsigned peers = __match_any_sync(am, key >> 20);
            if (lane == __ffs(peers) - 1)
                asm volatile("red.global.add.u32 [%0], %1;" ::"l"(p.hist + (key >> 20)),
                             "r"((uint32_t)__popc(peers))
                             : "memory");
        }
    }
    stamp(p.ts, 13);
    stamp(p.ts, 4);
    // grid barrier 2: every chunk's keys and histogram counts are out (its
    // __syncthreads also orders the shared-memory initialisation above)
    if (!grid_barrier(p.bar, (unsigned)nb * (gen + bi + 2u), p.status, p.limit_ns, ctl, false))
        return false;
    // every CTA has read gen (at the launch start): the next launch's
    if (last && b == 0 && tid == 0) *reinterpret_cast<volatile unsigned*>(p.epoch) = gen + bi + 2u;

    // ------------------------------------------------ P3: selection, then stage 2
    if (!select_items(p, ctl, area, nb, b, cb0, nch)) return false;
    const int m = ctl.n_items;  // every item is known before Stage 2 starts
    if (p.member) {  // a batch's union mask: record this token's share, no Stage 2
        for (int i = tid; i < m; i += kNT) atomicOr(p.member + ctl.item[i], 1u << p.token);
        stamp(p.ts, 5);
        return true;
    }
    if (tid == 0) stamp_here(p.ts, 5);
    __syncthreads();
    Stage2Args a;
    a.gateup = p.gateup;
    a.down_t = p.down_t;
    a.y = p.y;
    a.hch = p.debug ? p.hch : nullptr;
    a.status = p.status;
    a.d = d;
    a.F = F;
    a.n_gu = p.n_gu;
    a.n_d = p.n_d;
    a.n_a = p.n_a;
    a.limit_ns = p.limit_ns;
    a.ts = p.ts;
    if (wid != kSelectorWarp) stage2_roles<CPT, WQ>(a, ctl, area, m);
    stage2_join(a, ctl);
    return !*reinterpret_cast<volatile int*>(&ctl.abort);
}

// The decode step: one layer per launch.
template <int CPT, int WQ>
__global__ void __launch_bounds__(kNT, 1) k_prox_fused(const FusedParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Ctl& ctl = *reinterpret_cast<Ctl*>(smem_raw);
    uint8_t* area = smem_raw + ctl_bytes();  // phase-dependent union
    if (threadIdx.x == 0) {
        ctl.abort = 0;
        ctl.epoch = *reinterpret_cast<volatile unsigned*>(p.epoch);
    }
    __syncthreads();
    fused_step<CPT, WQ>(p, ctl, area, ctl.epoch, 0u, true);
}

// A stack of layers in one launch: layer l takes x_l = bf16(RMSNorm(x_{l-1}
// + y_{l-1})) (l > 0; computed inside its own step) and writes y_l; a grid
// barrier between layers makes y_{l-1} complete before layer l reads it.
// Each layer's parameters are the base parameters with that layer's
// weights and buffers, copied into shared memory for its step.  Layer l's
// step barriers are number gen + 3l + 1 and + 2; the barrier in front of
// layer l > 0 is number gen + 3l.
template <int CPT, int WQ>
__global__ void __launch_bounds__(kNT, 1) k_prox_stack(const FusedParams base, const StackLayers sl) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Ctl& ctl = *reinterpret_cast<Ctl*>(smem_raw);
    uint8_t* area = smem_raw + ctl_bytes();
    const int tid = threadIdx.x, nb = gridDim.x;
    if (tid == 0) {
        ctl.abort = 0;
        ctl.epoch = *reinterpret_cast<volatile unsigned*>(base.epoch);
    }
    __syncthreads();
    const unsigned gen = ctl.epoch;
    for (int l = 0; l < sl.n; ++l) {
        const unsigned bi = 3u * (unsigned)l;
        if (l > 0 && !grid_barrier(base.bar, (unsigned)nb * (gen + bi), base.status, base.limit_ns,
                                   ctl, false))
            return;
        if (tid == 0) {
            FusedParams q = base;
            const StackLayer& ly = sl.layer[l];
            q.codes = ly.codes;
            q.scales = ly.scales;
            q.gateup = ly.gateup;
            q.down_t = ly.down_t;
            q.y = sl.ys + (size_t)l * base.d;
            if (l == 0) {
                q.x = sl.x0;
                q.x_prev = nullptr;
            } else {
                q.x = nullptr;
                q.x_prev = l == 1 ? sl.x0 : sl.xs + (size_t)(l - 1) * base.d;
                q.y_prev = sl.ys + (size_t)(l - 1) * base.d;
                q.x_out = sl.xs + (size_t)l * base.d;
            }
            ctl.sp = q;
        }
        __syncthreads();
        if (!fused_step<CPT, WQ>(ctl.sp, ctl, area, gen, bi, l + 1 == sl.n)) return;
    }
}

// Stage 1 of several tokens at once (a batch's masks): the grid splits into
// groups of mg.gsize CTAs, group t runs token t's step in mask-only mode on
// its own x, y row, histogram, proxy partials, score keys and barrier word
// (mg.scratch + t mg.stride, mg.gbar[t], the latter zero at launch).
template <int CPT, int WQ>
__global__ void __launch_bounds__(kNT, 1) k_prox_masks(const FusedParams base, const MaskGroups mg) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Ctl& ctl = *reinterpret_cast<Ctl*>(smem_raw);
    uint8_t* area = smem_raw + ctl_bytes();
    const int tk = (int)blockIdx.x / base.gsize;
    if (threadIdx.x == 0) {
        ctl.abort = 0;
        FusedParams q = base;
        uint8_t* sc = mg.scratch + (size_t)tk * mg.stride;
        q.x = base.x + (size_t)tk * base.d;
        q.y = base.y + (size_t)tk * base.d;
        q.hist = reinterpret_cast<uint32_t*>(sc);
        q.part = reinterpret_cast<float2*>(sc + mg.part_off);
        q.skey = reinterpret_cast<uint32_t*>(sc + mg.skey_off);
        q.bar = mg.gbar + tk;
        q.token = mg.token0 + tk;
        ctl.sp = q;
    }
    __syncthreads();
    fused_step<CPT, WQ, true>(ctl.sp, ctl, area, 0u, 0u, false);
}

// Dense baseline: Stage 2 over every channel, CTA i taking [F i/n, F (i+1)/n)
// (all items known and confirmed from the start).
template <int CPT, int WQ>
__global__ void __launch_bounds__(kNT, 1) k_dense(const Stage2Args a, const uint16_t* x) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Ctl& ctl = *reinterpret_cast<Ctl*>(smem_raw);
    uint8_t* area = smem_raw + ctl_bytes();
    const int tid = threadIdx.x;
    stamp(a.ts, 0);
    const int c0 = chunk_begin(a.F, blockIdx.x, gridDim.x);
    const int n = chunk_begin(a.F, blockIdx.x + 1, gridDim.x) - c0;  // <= kMaxChunk
    for (int i = tid; i < a.d / 8; i += kNT)
        reinterpret_cast<uint4*>(area)[i] = __ldg(reinterpret_cast<const uint4*>(x) + i);
    for (int i = tid; i < kMaxItems; i += kNT) {
        ctl.item[i] = c0 + i;
        ctl.hready[i] = 0;
    }
    if (tid == 0) {
        ctl.abort = 0;
        ctl.n_items = n;
        stage2_init(ctl, a.n_gu, a.n_d);
        fence_mbar_init();
    }
    __syncthreads();
    if ((tid >> 5) != kSelectorWarp) stage2_roles<CPT, WQ>(a, ctl, area, n);
    stage2_join(a, ctl);
}

// Debug: the channel list and h in list order from the per-channel arrays.
__global__ void k_gather_h(const int* idx_list, const float* hch, int k, int32_t* idx_out,
                           float* h_out) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < k; i += gridDim.x * blockDim.x) {
        const int c = idx_list[i];
        if (idx_out) idx_out[i] = c;
        if (h_out) h_out[i] = hch[c];
    }
}

// ------------------------------------------------------------ host side
struct Ring {
    int n_gu, n_d, n_a;
};

size_t area_budget() { return kSmemLimit - ctl_bytes(); }

// Stage-2 rings after x (stage2_x_bytes): gate|up stages (one row each) up to
// kGuRingBytes (bf16) or kGuRingBytesQ (int8, int4) and kMaxStages, consumed by
// n_a = min(stages, kPassAWarps) pass-A warps (the stage count rounded down
// to a multiple of n_a), then W_down^T stages up to kDRingBytes, both within
// the shared memory left; for codes, the pass-B slots of n_d items (8, 4 or
// 2, at most a third of the area) come first.  The bf16 caps keep ~160 KB
// in flight per SM:
// enough to saturate HBM, and every extra byte in flight only lengthens the
// queues that the channel selection's loads wait in.  Rows of int8 are half
// as long, so their ring holds more of them; int4 rows a quarter, so theirs
// is kMaxStages deep (~66 KB at d = 4096).
// x in the Stage-2 area: bf16 (2 d bytes), and for codes also fp32 (4 d).
size_t stage2_x_bytes(int d, int wq) { return (size_t)(wq ? 6 : 2) * d; }

Ring ring_for(int d, int wq) {
    const size_t budget = area_budget() - stage2_x_bytes(d, wq);
    const size_t gu = gu_row_bytes(d, wq);
    Ring r{0, 0, 0};
    size_t dbytes = 0;  // the W_down^T stream
    if (wq) {
        // codes: n_d = items each pass-B thread streams ahead (8, 4 or 2),
        // taking at most a third of the area
        const size_t per = self_item_bytes(d, wq);
        r.n_d = 8;
        while (r.n_d > 2 && (size_t)r.n_d * per > budget / 3) r.n_d /= 2;
        dbytes = (size_t)r.n_d * per;
    }
    const size_t room = budget > dbytes ? budget - dbytes : 0;
    r.n_gu = (int)(min(wq ? room : budget * 2 / 3, wq ? kGuRingBytesQ : kGuRingBytes) / gu);
    if (r.n_gu > kMaxStages) r.n_gu = kMaxStages;
    if (r.n_gu < 1) r.n_gu = 1;
    r.n_a = r.n_gu < kPassAWarps ? r.n_gu : kPassAWarps;
    r.n_gu -= r.n_gu % r.n_a;
    if (!wq) {
        const size_t dd = down_row_bytes(d, 0);
        const size_t left = budget > (size_t)r.n_gu * gu ? budget - (size_t)r.n_gu * gu : 0;
        r.n_d = (int)(min(left, kDRingBytes) / dd);
        if (r.n_d > kMaxStages) r.n_d = kMaxStages;
        if (r.n_d < 1 && left >= dd) r.n_d = 1;
    }
    return r;
}

size_t ring_bytes(int d, int wq, const Ring& r) {
    return stage2_x_bytes(d, wq) + (size_t)r.n_gu * gu_row_bytes(d, wq) +
           (size_t)r.n_d * (wq ? self_item_bytes(d, wq) : down_row_bytes(d, wq));
}

template <typename K>
cudaError_t set_smem(K kern) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
}

}  // namespace

ProxyGeom proxy_geometry(int F, int kx, int num_blocks, bool any_width) {
    // Tiles of W = 16 tpr channels (tpr threads per proxy row), T tiles x S
    // slices <= blocks.  No fit (more 1024-channel tiles than blocks):
    // tiles = 0.
    //  * a whole-grid step: W = 256, 512 or 1024 (a row is whole half-warps);
    //    minimise the bytes of the busiest CTA, then prefer fewer slices
    //    (less partial traffic);
    //  * any_width (a group of a few CTAs per token): any tpr in 8..64;
    //    minimise the kept rows per thread of the busiest CTA (its slice's
    //    rows over its kNT / tpr row-lanes), then fewer slices.  On the
    //    whole grid this measured slower (a step of the Llama-3-8B layer:
    //    688-channel tiles, 48.6 against 47.0 us); in groups of 18 CTAs it
    //    keeps every CTA busy (800-channel tiles: 18 instead of 14 CTAs).
    const int Fp = padded_ff(F);
    ProxyGeom best{0, 1, 1024};
    long long best_cost = -1;
    for (int tpr = any_width ? 8 : 16; tpr <= 64; tpr += any_width ? 1 : tpr) {
        const int W = 16 * tpr;
        const int T = (Fp + W - 1) / W;
        if (T > num_blocks) continue;
        int S = num_blocks / T;
        if (S > kMaxSlices) S = kMaxSlices;
        if (S > kx) S = kx;
        if (S < 1) S = 1;
        const long long rows = (kx + S - 1) / S;
        const long long cost = any_width ? (rows + kNT / tpr - 1) / (kNT / tpr) : (long long)min(W, Fp) * rows;
        if (best_cost < 0 || cost < best_cost || (cost == best_cost && S < best.slices)) {
            best_cost = cost;
            best = {T, S, W};
        }
    }
    return best;
}

cudaError_t fused_configure() {
    cudaError_t e = cudaSuccess;
    auto all = [&](auto k1, auto k2, auto k4, auto k8) {
        if (e == cudaSuccess) e = set_smem(k1);
        if (e == cudaSuccess) e = set_smem(k2);
        if (e == cudaSuccess) e = set_smem(k4);
        if (e == cudaSuccess) e = set_smem(k8);
    };
    all(k_prox_fused<1, 0>, k_prox_fused<2, 0>, k_prox_fused<4, 0>, k_prox_fused<8, 0>);
    all(k_prox_fused<1, 1>, k_prox_fused<2, 1>, k_prox_fused<4, 1>, k_prox_fused<8, 1>);
    all(k_prox_fused<1, 2>, k_prox_fused<2, 2>, k_prox_fused<4, 2>, k_prox_fused<8, 2>);
    all(k_prox_masks<1, 0>, k_prox_masks<2, 0>, k_prox_masks<4, 0>, k_prox_masks<8, 0>);
    all(k_prox_stack<1, 0>, k_prox_stack<2, 0>, k_prox_stack<4, 0>, k_prox_stack<8, 0>);
    all(k_prox_stack<1, 1>, k_prox_stack<2, 1>, k_prox_stack<4, 1>, k_prox_stack<8, 1>);
    all(k_prox_stack<1, 2>, k_prox_stack<2, 2>, k_prox_stack<4, 2>, k_prox_stack<8, 2>);
    all(k_dense<1, 0>, k_dense<2, 0>, k_dense<4, 0>, k_dense<8, 0>);
    all(k_dense<1, 1>, k_dense<2, 1>, k_dense<4, 1>, k_dense<8, 1>);
    all(k_dense<1, 2>, k_dense<2, 2>, k_dense<4, 2>, k_dense<8, 2>);
    return e;
}

size_t fused_smem_bytes() { return kSmemLimit; }

int fused_threads() { return kNT; }

int fused_max_chunk() { return kMaxChunk; }

int fused_max_blocks() { return kMaxBlocks; }

bool fused_fits(int d, int F) {
    // P0: x (2 d) + kept list (4 d) + histograms; P1 adds the cp.async ring
    // (the running-total table reuses it); P3: the Stage-2 rings.
    const size_t p01 = (size_t)6 * d + 4096 + (size_t)16 * kRing * kNT;
    const Ring r = ring_for(d, 0);  // the bf16 rings are the larger
    // the channel selection (every CTA): x, three digit histograms and
    // every channel's score key
    const size_t sel = (size_t)2 * d + (size_t)4 * (kHistBins + 512) + (size_t)4 * padded_ff(F);
    return p01 <= area_budget() && ring_bytes(d, 0, r) <= area_budget() &&
           ring_bytes(d, 1, ring_for(d, 1)) <= area_budget() &&
           ring_bytes(d, 2, ring_for(d, 2)) <= area_budget() && sel <= area_budget() &&
           r.n_gu >= 1 && r.n_d >= 1 && d / 8 <= kXGroups * kNT;
}

namespace {
template <int CPT>
cudaError_t launch_fused_t(const cudaLaunchConfig_t& cfg, const FusedParams& p) {
    switch (p.wq) {
        case 0: return cudaLaunchKernelEx(&cfg, k_prox_fused<CPT, 0>, p);
        case 1: return cudaLaunchKernelEx(&cfg, k_prox_fused<CPT, 1>, p);
        case 2: return cudaLaunchKernelEx(&cfg, k_prox_fused<CPT, 2>, p);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace

namespace {
FusedParams make_params(const FusedLaunch& L) {
    FusedParams p;
    p.codes = L.codes;
    p.scales = L.scales;
    p.gateup = static_cast<const uint8_t*>(L.gateup);
    p.down_t = static_cast<const uint8_t*>(L.down_t);
    p.wq = L.wq;
    p.d = L.d;
    p.F = L.F;
    p.Fp = padded_ff(L.F);
    p.x = L.x;
    p.y = L.y;
    p.kx = L.kx;
    p.k = L.k;
    p.bw = L.bw;
    p.dnorm = L.dnorm;
    p.x_prev = L.x_prev;
    p.y_prev = L.y_prev;
    p.x_out = L.x_out;
    p.eps = L.eps;
    const ProxyGeom geo = proxy_geometry(L.F, L.kx, L.num_blocks, false);
    p.tiles = geo.tiles;
    p.slices = geo.slices;
    p.tile_w = geo.tile_w;
    p.status = L.ws->status;
    p.bar = L.ws->bar;
    p.epoch = L.ws->bar + 1;
    p.hist = L.ws->hist;
    p.part = L.ws->part;
    p.skey = L.ws->skey;
    p.idx_list = L.ws->idx_list;
    p.hch = L.ws->hch;
    p.kept_out = L.kept_out;
    p.scores_out = L.scores_out;
    p.debug = (L.idx_out || L.h_out) ? 1 : 0;
    const Ring r = ring_for(L.d, L.wq);
    p.n_gu = r.n_gu;
    p.n_d = r.n_d;
    p.n_a = r.n_a;
    p.limit_ns = L.limit_ns;
    p.inject = L.inject;
    p.ts = L.ts;
    p.member = L.member;
    p.token = L.token;
    p.gsize = 0;
    return p;
}

cudaLaunchConfig_t coop_config(int blocks, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kNT);
    cfg.dynamicSmemBytes = kSmemLimit;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <int CPT>
cudaError_t launch_stack_t(const cudaLaunchConfig_t& cfg, const FusedParams& p, const StackLayers& sl) {
    switch (p.wq) {
        case 0: return cudaLaunchKernelEx(&cfg, k_prox_stack<CPT, 0>, p, sl);
        case 1: return cudaLaunchKernelEx(&cfg, k_prox_stack<CPT, 1>, p, sl);
        case 2: return cudaLaunchKernelEx(&cfg, k_prox_stack<CPT, 2>, p, sl);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace

cudaError_t launch_fused(const FusedLaunch& L, cudaStream_t stream) {
    if (L.num_blocks < 1 || L.num_blocks > kMaxBlocks) return cudaErrorInvalidValue;
    const FusedParams p = make_params(L);
    if (p.tiles < 1) return cudaErrorInvalidValue;  // a proxy tile per CTA at most
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = coop_config(L.num_blocks, stream, attr);
    const int nchunk = L.d / 8;
    cudaError_t e;
    if (nchunk <= kPassB) e = launch_fused_t<1>(cfg, p);
    else if (nchunk <= 2 * kPassB) e = launch_fused_t<2>(cfg, p);
    else if (nchunk <= 4 * kPassB) e = launch_fused_t<4>(cfg, p);
    else e = launch_fused_t<8>(cfg, p);
    if (e == cudaSuccess && p.debug) {
        k_gather_h<<<(L.k + 255) / 256, 256, 0, stream>>>(L.ws->idx_list, L.ws->hch, L.k,
                                                         L.idx_out, L.h_out);
        e = cudaGetLastError();
    }
    return e;
}

cudaError_t launch_stack(const FusedLaunch& L, const StackLayers& sl, cudaStream_t stream) {
    if (L.num_blocks < 1 || L.num_blocks > kMaxBlocks || sl.n < 1 || sl.n > kMaxStack)
        return cudaErrorInvalidValue;
    FusedParams p = make_params(L);
    if (p.tiles < 1) return cudaErrorInvalidValue;
    p.debug = 0;
    p.kept_out = nullptr;
    p.scores_out = nullptr;
    p.ts = nullptr;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = coop_config(L.num_blocks, stream, attr);
    const int nchunk = L.d / 8;
    if (nchunk <= kPassB) return launch_stack_t<1>(cfg, p, sl);
    if (nchunk <= 2 * kPassB) return launch_stack_t<2>(cfg, p, sl);
    if (nchunk <= 4 * kPassB) return launch_stack_t<4>(cfg, p, sl);
    return launch_stack_t<8>(cfg, p, sl);
}

MaskGroupGeom mask_group_geometry(int d, int F, int k, int ntok, int num_blocks) {
    MaskGroupGeom g{};
    if (ntok < 2) return g;
    const int gsize = num_blocks / ntok;
    const int kx = (d + 1) / 2;  // the input keep count of a step (keep fraction 0.5)
    if (gsize < 4 || (k + gsize - 1) / gsize > kMaxItems) return g;
    const int Fp = padded_ff(F);
    // the proxy needs a CTA per tile of up to 1024 channels
    if ((Fp + 1023) / 1024 > gsize) return g;
    const ProxyGeom geo = proxy_geometry(F, kx, gsize, true);
    auto a256 = [](size_t v) { return (v + 255) / 256 * 256; };
    g.gsize = gsize;
    g.part_off = a256((size_t)kHistWords * 4);
    g.skey_off = g.part_off + a256((size_t)geo.slices * Fp * 8);
    g.stride = g.skey_off + a256((size_t)Fp * 4);
    return g;
}

cudaError_t launch_masks(const FusedLaunch& L, int ntok, int token0, uint8_t* scratch,
                         unsigned* gbar, cudaStream_t stream) {
    const MaskGroupGeom g = mask_group_geometry(L.d, L.F, L.k, ntok, L.num_blocks);
    if (g.gsize == 0 || !L.member || L.wq || L.bw) return cudaErrorInvalidValue;
    FusedParams p = make_params(L);
    const ProxyGeom geo = proxy_geometry(L.F, L.kx, g.gsize, true);
    if (geo.tiles < 1) return cudaErrorInvalidValue;
    p.tiles = geo.tiles;
    p.slices = geo.slices;
    p.tile_w = geo.tile_w;
    p.gsize = g.gsize;
    p.debug = 0;
    p.kept_out = nullptr;
    p.scores_out = nullptr;
    p.ts = nullptr;
    MaskGroups mg;
    mg.scratch = scratch;
    mg.stride = g.stride;
    mg.part_off = g.part_off;
    mg.skey_off = g.skey_off;
    mg.gbar = gbar;
    mg.token0 = token0;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = coop_config(ntok * g.gsize, stream, attr);
    const int nchunk = L.d / 8;
    const int cpt = nchunk <= kPassB ? 1 : nchunk <= 2 * kPassB ? 2 : nchunk <= 4 * kPassB ? 4 : 8;
    switch (cpt) {
        case 1: return cudaLaunchKernelEx(&cfg, k_prox_masks<1, 0>, p, mg);
        case 2: return cudaLaunchKernelEx(&cfg, k_prox_masks<2, 0>, p, mg);
        case 4: return cudaLaunchKernelEx(&cfg, k_prox_masks<4, 0>, p, mg);
        default: return cudaLaunchKernelEx(&cfg, k_prox_masks<8, 0>, p, mg);
    }
}

cudaError_t launch_dense(const void* gateup, const void* down_t, int wq, const uint16_t* x, int d,
                         int F, float* y, int* status, int num_blocks, long long limit_ns,
                         uint64_t* ts, cudaStream_t stream) {
    if (num_blocks < 1 || num_blocks > kMaxBlocks) return cudaErrorInvalidValue;
    Stage2Args a;
    a.gateup = static_cast<const uint8_t*>(gateup);
    a.down_t = static_cast<const uint8_t*>(down_t);
    a.y = y;
    a.hch = nullptr;
    a.status = status;
    a.d = d;
    a.F = F;
    const Ring r = ring_for(d, wq);
    a.n_gu = r.n_gu;
    a.n_d = r.n_d;
    a.n_a = r.n_a;
    a.limit_ns = limit_ns;
    a.ts = ts;
    const int nchunk = d / 8;
    const int cpt = nchunk <= kPassB ? 1 : nchunk <= 2 * kPassB ? 2 : nchunk <= 4 * kPassB ? 4 : 8;
    auto go = [&](auto kern) {
        kern<<<num_blocks, kNT, kSmemLimit, stream>>>(a, x);
        return cudaGetLastError();
    };
    if (wq < 0 || wq > 2) return cudaErrorInvalidValue;
    switch (cpt * 4 + wq) {
        case 4: return go(k_dense<1, 0>);
        case 5: return go(k_dense<1, 1>);
        case 6: return go(k_dense<1, 2>);
        case 8: return go(k_dense<2, 0>);
        case 9: return go(k_dense<2, 1>);
        case 10: return go(k_dense<2, 2>);
        case 16: return go(k_dense<4, 0>);
        case 17: return go(k_dense<4, 1>);
        case 18: return go(k_dense<4, 2>);
        case 32: return go(k_dense<8, 0>);
        case 33: return go(k_dense<8, 1>);
        default: return go(k_dense<8, 2>);
    }
}

}  // namespace prox
