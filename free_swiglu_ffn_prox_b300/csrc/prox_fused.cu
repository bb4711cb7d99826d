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
constexpr int kUnroll = 8;               // proxy rows in flight per thread
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
    float fmax_part[kNT / 32];
    int abort;
    int chan[kMaxChan];
};

constexpr size_t ctl_bytes() { return (sizeof(Ctl) + 127) / 128 * 128; }

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
__device__ __forceinline__ unsigned atom_add_release_gpu(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.add.release.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier for co-resident CTAs without a reset between uses: CTA 0
// adds 2^31 - (n - 1), every other CTA adds 1, so each completed barrier
// flips bit 31 and leaves the low bits unchanged.  Returns false (and
// records PROX_ERR_TIMEOUT) if the flip does not come within limit_ns.
__device__ bool grid_barrier(unsigned* bar, int* status, long long limit_ns, Ctl& ctl,
                             bool skip_arrive) {
    __syncthreads();
    if (threadIdx.x == 0) {
        bool ok = true;
        if (!skip_arrive) {
            __threadfence();
            const unsigned inc = blockIdx.x == 0 ? 0x80000000u - (gridDim.x - 1) : 1u;
            const unsigned old = atom_add_release_gpu(bar, inc);
            const uint64_t t0 = global_timer_ns();
            for (uint32_t it = 0;; ++it) {
                if (((ld_acquire_gpu(bar) ^ old) & 0x80000000u) != 0) break;
                if ((it & 15u) == 15u && (long long)(global_timer_ns() - t0) > limit_ns) {
                    ok = false;
                    break;
                }
            }
            __threadfence();
        } else {
            ok = false;
        }
        if (!ok) {
            record_status(status, PROX_ERR_TIMEOUT);
            ctl.abort = 1;
        }
    }
    __syncthreads();
    return ctl.abort == 0;
}

// Exclusive scan of one value per thread over the block; also the total.
__device__ __forceinline__ uint32_t block_scan(uint32_t v, Ctl& ctl, uint32_t& total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint32_t s = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += t;
    }
    if (lane == 31) ctl.warp_tot[wid] = s;
    __syncthreads();
    if (wid == 0) {
        const uint32_t w = lane < kNT / 32 ? ctl.warp_tot[lane] : 0u;
        uint32_t ws = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, ws, o);
            if (lane >= o) ws += t;
        }
        if (lane < kNT / 32) ctl.warp_tot[lane] = ws - w;
        if (lane == kNT / 32 - 1) ctl.warp_tot[kNT / 32] = ws;
    }
    __syncthreads();
    const uint32_t excl = ctl.warp_tot[wid] + s - v;
    total = ctl.warp_tot[kNT / 32];
    __syncthreads();
    return excl;
}

// h[bin] += 1 for the active lanes, one atomic per distinct bin in the warp.
// Every lane of the warp must call it.
__device__ __forceinline__ void hist_add_smem(uint32_t* h, uint32_t bin, bool active) {
    const unsigned m = __ballot_sync(0xffffffffu, active);
    if (active) {
        const unsigned peers = __match_any_sync(m, bin);
        if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&h[bin], (uint32_t)__popc(peers));
    }
}

__device__ __forceinline__ void hist_add_global(uint32_t* h, uint32_t bin, bool active) {
    const unsigned m = __ballot_sync(0xffffffffu, active);
    if (active) {
        const unsigned peers = __match_any_sync(m, bin);
        if ((threadIdx.x & 31) == __ffs(peers) - 1)
            asm volatile("red.global.add.u32 [%0], %1;" ::"l"(h + bin), "r"((uint32_t)__popc(peers))
                         : "memory");
    }
}

// Given a histogram h[nbins] of digits and krem >= 1 with sum(h) >= krem,
// finds the digit b with sum(h[b+1..]) < krem <= sum(h[b..]) and returns
// (b, krem - sum(h[b+1..])) in ctl.sel[0..1] for every thread.
__device__ void select_bin(const uint32_t* h, int nbins, uint32_t krem, Ctl& ctl) {
    const int per = (nbins + kNT - 1) / kNT;
    // thread t owns the bins [nbins - (t+1) per, nbins - t per) (from the top)
    const int hi = nbins - threadIdx.x * per;
    const int lo = max(hi - per, 0);
    uint32_t sum = 0;
    for (int b = lo; b < hi; ++b) sum += h[b];
    uint32_t total;
    const uint32_t above = block_scan(hi > 0 ? sum : 0u, ctl, total);  // count in bins >= hi
    if (hi > 0 && above < krem && above + sum >= krem) {
        uint32_t acc = above;
        for (int b = hi - 1; b >= lo; --b) {
            if (acc + h[b] >= krem) {
                ctl.sel[0] = (uint32_t)b;
                ctl.sel[1] = krem - acc;
                break;
            }
            acc += h[b];
        }
    }
    __syncthreads();
}

// Emits, in ascending index order, the indices i < n whose key(i) > T plus
// the first r (lowest) with key(i) == T.  emit(pos, i) is called for each.
template <typename KeyFn, typename Emit>
__device__ void compact_topk(int n, uint32_t T, uint32_t r, KeyFn key, Emit emit, Ctl& ctl) {
    const int per = (n + kNT - 1) / kNT;
    const int i0 = min(n, (int)threadIdx.x * per), i1 = min(n, i0 + per);
    uint32_t gt = 0, eq = 0;
    for (int i = i0; i < i1; ++i) {
        const uint32_t kk = key(i);
        gt += kk > T;
        eq += kk == T;
    }
    uint32_t tg, te;
    const uint32_t pg = block_scan(gt, ctl, tg);
    const uint32_t pe = block_scan(eq, ctl, te);
    uint32_t pos = pg + min(pe, r);
    uint32_t tie = pe;
    for (int i = i0; i < i1; ++i) {
        const uint32_t kk = key(i);
        bool keep = kk > T;
        if (kk == T) {
            keep = tie < r;
            ++tie;
        }
        if (keep) emit(pos++, i);
    }
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

__device__ __forceinline__ uint4 ldg_stream(const void* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
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
    for (int i = threadIdx.x; i < nchunk; i += kNT)
        reinterpret_cast<uint4*>(xs)[i] = __ldg(reinterpret_cast<const uint4*>(a.x) + i);
    __syncthreads();

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

// ------------------------------------------------------------ fused kernel
template <int CPT>
__global__ void __launch_bounds__(kNT, 1) k_prox_fused(const FusedParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Ctl& ctl = *reinterpret_cast<Ctl*>(smem_raw);
    uint8_t* area = smem_raw + ctl_bytes();  // phase-dependent union
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nb = gridDim.x, b = blockIdx.x;
    const int d = p.d, F = p.F, Fp = p.Fp;
    if (tid == 0) ctl.abort = 0;
    stamp(p.ts, 0);

    // ------------------------------------------------ P0: input sparsity
    uint16_t* xs = reinterpret_cast<uint16_t*>(area);                       // [d]
    uint32_t* kept = reinterpret_cast<uint32_t*>(area + (size_t)2 * d);      // [d]
    uint32_t* hsm = kept + d;                                                // [kHistBins]
    for (int i = tid; i < d / 8; i += kNT)
        reinterpret_cast<uint4*>(xs)[i] = __ldg(reinterpret_cast<const uint4*>(p.x) + i);
    if (b == 0) {
        for (int i = tid; i < d; i += kNT) p.y[i] = 0.0f;
        for (int i = tid; i < kHistBins; i += kNT) p.hist[i] = 0u;
    }
    for (int i = tid; i < 256; i += kNT) hsm[i] = 0u;
    __syncthreads();
    int shift;
    {
        uint32_t mk = 0;
        for (int i = tid; i < d; i += kNT) mk = max(mk, (uint32_t)(xs[i] & 0x7fffu));
        mk = __reduce_max_sync(0xffffffffu, mk);
        if (lane == 0) ctl.warp_tot[wid] = mk;
        __syncthreads();
        mk = 0;
        for (int w = 0; w < kNT / 32; ++w) mk = max(mk, ctl.warp_tot[w]);
        shift = 0;
        if (mk != 0) {
            int ex;
            frexpf(__uint_as_float(mk << 16), &ex);  // max|x| in [2^(ex-1), 2^ex)
            shift = 15 - ex;
        }
        __syncthreads();
    }
    // digit 1: |x| bits 14..7
    const int xrounds = (d + kNT - 1) / kNT;
    for (int e = 0; e < xrounds; ++e) {
        const int i = tid + e * kNT;
        const uint32_t kk = i < d ? (xs[i] & 0x7fffu) : 0u;
        hist_add_smem(hsm, kk >> 7, i < d);
    }
    __syncthreads();
    select_bin(hsm, 256, (uint32_t)p.kx, ctl);
    const uint32_t xb1 = ctl.sel[0], xk1 = ctl.sel[1];
    for (int i = tid; i < 128; i += kNT) hsm[i] = 0u;
    __syncthreads();
    for (int e = 0; e < xrounds; ++e) {
        const int i = tid + e * kNT;
        const uint32_t kk = i < d ? (xs[i] & 0x7fffu) : 0u;
        hist_add_smem(hsm, kk & 127u, i < d && (kk >> 7) == xb1);
    }
    __syncthreads();
    select_bin(hsm, 128, xk1, ctl);
    const uint32_t xT = (xb1 << 7) | ctl.sel[0], xr = ctl.sel[1];
    compact_topk(
        d, xT, xr, [&](int i) { return (uint32_t)(xs[i] & 0x7fffu); },
        [&](uint32_t pos, int j) {
            const float xv = ldexpf(__uint_as_float((uint32_t)xs[j] << 16), shift);
            kept[pos] = ((uint32_t)j << 16) | __half_as_ushort(__float2half_rn(xv));
            if (b == 0 && p.kept_out) p.kept_out[pos] = j;
        },
        ctl);
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
        // running totals, [R][16][tpr] float2: channel cu * 16 + t of row-lane
        // rl at (rl * 16 + t) * tpr + cu, so a warp's lanes (consecutive cu)
        // touch consecutive 8-byte words
        float2* tot = reinterpret_cast<float2*>(hsm + kHistBins);
        if (active)
            for (int t = 0; t < 16; ++t) tot[((size_t)rl * 16 + t) * tpr + cu] = make_float2(0.0f, 0.0f);
        float ag[16], au[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) ag[t] = au[t] = 0.0f;
        int cur_g = -1;
        auto flush = [&]() {
            if (cur_g < 0) return;
            const uint4* src = reinterpret_cast<const uint4*>(p.scales + (size_t)cur_g * Fp + c0 + cu * 16);
            float2* dst = tot + (size_t)rl * 16 * tpr + cu;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 s4 = __ldg(src + v);
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
        if (active) {
            const uint64_t pol = policy_evict_first();
            const uint8_t* colbase = p.codes + c0 + cu * 16;
            for (int q0 = r0 + rl; q0 < r1; q0 += R * kUnroll) {
                uint4 w[kUnroll];
                uint32_t kp[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int q = q0 + u * R;
                    kp[u] = 0;
                    w[u] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
                    if (q < r1) {
                        kp[u] = kept[q];
                        w[u] = ldg_stream(colbase + (size_t)(kp[u] >> 16) * Fp, pol);
                    }
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int q = q0 + u * R;
                    if (q < r1) {
                        const int g = (int)(kp[u] >> 23);  // j / 128
                        if (g != cur_g) {
                            flush();
                            cur_g = g;
                        }
                        const uint16_t xh = (uint16_t)(kp[u] & 0xffffu);
                        proxy_mac_word(w[u].x, xh, &ag[0], &au[0]);
                        proxy_mac_word(w[u].y, xh, &ag[4], &au[4]);
                        proxy_mac_word(w[u].z, xh, &ag[8], &au[8]);
                        proxy_mac_word(w[u].w, xh, &ag[12], &au[12]);
                    }
                }
            }
            flush();
        }
        __syncthreads();
        float2* out = p.part + (size_t)slice * Fp + c0;
        for (int cl = tid; cl < width; cl += kNT) {
            float g = 0.0f, u = 0.0f;
            const int cu_ = cl >> 4, t_ = cl & 15;
            for (int r = 0; r < R; ++r) {
                const float2 v = tot[((size_t)r * 16 + t_) * tpr + cu_];
                g += v.x;
                u += v.y;
            }
            out[cl] = make_float2(ldexpf(g, -shift), ldexpf(u, -shift));
        }
    }
    stamp(p.ts, 2);
    if (!grid_barrier(p.bar, p.status, p.limit_ns, ctl, p.inject == 1 && b == nb - 1)) return;
    stamp(p.ts, 3);

    // ------------------------------------------------ P2: scores + histogram
    {
        const int cb0 = (int)((long long)F * b / nb), cb1 = (int)((long long)F * (b + 1) / nb);
        for (int c00 = cb0; c00 < cb1; c00 += kNT) {
            const int c = c00 + tid;
            const bool act = c < cb1;
            uint32_t key = 0;
            if (act) {
                float g = 0.0f, u = 0.0f;
                for (int s = 0; s < p.slices; ++s) {
                    const float2 v = __ldcg(p.part + (size_t)s * Fp + c);
                    g += v.x;
                    u += v.y;
                }
                // |silu(g~) * u~|, silu(z) = z / (1 + e^-z)
                const float sc = fabsf(g / (1.0f + expf(-g)) * u);
                p.scores[c] = sc;
                if (p.scores_out) p.scores_out[c] = sc;
                key = __float_as_uint(sc);
            }
            hist_add_global(p.hist, key >> 20, act);
        }
    }
    stamp(p.ts, 4);
    if (!grid_barrier(p.bar, p.status, p.limit_ns, ctl, false)) return;
    stamp(p.ts, 5);

    // ------------------------------------------------ P3: exact top-k, this CTA's share
    int n_mine;
    {
        uint32_t* h = reinterpret_cast<uint32_t*>(area);                        // [kHistBins]
        float* sc = reinterpret_cast<float*>(area + kHistBins * sizeof(uint32_t)); // [F]
        for (int i = tid; i < kHistBins; i += kNT) h[i] = __ldcg(p.hist + i);
        for (int i = tid; i < F; i += kNT) sc[i] = __ldcg(p.scores + i);
        __syncthreads();
        select_bin(h, kHistBins, (uint32_t)p.k, ctl);
        const uint32_t b1 = ctl.sel[0], k1 = ctl.sel[1];
        for (int i = tid; i < kHistBins; i += kNT) h[i] = 0u;
        __syncthreads();
        const int frounds = (F + kNT - 1) / kNT;
        for (int e = 0; e < frounds; ++e) {
            const int i = tid + e * kNT;
            const uint32_t kk = i < F ? __float_as_uint(sc[i]) : 0u;
            hist_add_smem(h, (kk >> 9) & 2047u, i < F && (kk >> 20) == b1);
        }
        __syncthreads();
        select_bin(h, kHistBins, k1, ctl);
        const uint32_t b12 = (b1 << 11) | ctl.sel[0], k2 = ctl.sel[1];
        for (int i = tid; i < 512; i += kNT) h[i] = 0u;
        __syncthreads();
        for (int e = 0; e < frounds; ++e) {
            const int i = tid + e * kNT;
            const uint32_t kk = i < F ? __float_as_uint(sc[i]) : 0u;
            hist_add_smem(h, kk & 511u, i < F && (kk >> 9) == b12);
        }
        __syncthreads();
        select_bin(h, 512, k2, ctl);
        const uint32_t T = (b12 << 9) | ctl.sel[0], r = ctl.sel[1];
        const int p0 = (int)((long long)p.k * b / nb), p1 = (int)((long long)p.k * (b + 1) / nb);
        n_mine = p1 - p0;
        compact_topk(
            F, T, r, [&](int i) { return __float_as_uint(sc[i]); },
            [&](uint32_t pos, int c) {
                if ((int)pos >= p0 && (int)pos < p1) {
                    ctl.chan[pos - p0] = c;
                    if (p.idx_out) p.idx_out[pos] = c;
                }
            },
            ctl);
        __syncthreads();
    }

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
    const int Fp = padded_ff(F);
    const int units = Fp / 16;
    ProxyGeom best{1, 1, units * 16};
    long long best_cost = -1;
    for (int T = 1; T <= num_blocks && T <= units; ++T) {
        int S = num_blocks / T;
        if (S > kMaxSlices) S = kMaxSlices;
        if (S > kx) S = kx;
        if (S < 1) S = 1;
        const int wu = (units + T - 1) / T;
        if (wu * 16 > 16 * kNT) continue;  // a row segment needs at most one thread per 16 bytes
        const long long cost = (long long)wu * 16 * ((kx + S - 1) / S);
        if (best_cost < 0 || cost < best_cost || (cost == best_cost && S < best.slices)) {
            best_cost = cost;
            best = {T, S, wu * 16};
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
    const size_t p01 = (size_t)6 * d + kHistBins * 4 + (size_t)8 * 16 * kNT;
    const size_t p3 = (size_t)kHistBins * 4 + (size_t)4 * F;
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
