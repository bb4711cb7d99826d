// prox_internal.cuh -- shared device helpers and launcher declarations for
// libprox (sm_103a).  Inline PTX for mbarriers and bulk (TMA) copies, the
// bounded waits every kernel uses, and the workspace layout.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "prox.h"

namespace prox {

constexpr int kMaxDModel = 16384;
constexpr int kMaxDff = 32768;
constexpr int kGroup = 128;       // proxy quantization group along d_model
constexpr int kChanAlign = 64;    // Fp = d_ff rounded up to this
constexpr long long kWaitLimitNs = 2000000000LL;  // 2 s per bounded wait

inline int padded_ff(int d_ff) { return (d_ff + kChanAlign - 1) / kChanAlign * kChanAlign; }

constexpr int kMaxSlices = 16;   // proxy row slices (partial sums per channel)
constexpr int kHistWords = 2048; // score histogram (top 11 bits of the bit pattern)
constexpr int kMaxGrid = 256;    // CTAs of the fused kernel (one per SM)
constexpr size_t kControlBytes = 2048;

// Workspace carve-out (offsets in bytes, each 256-aligned).  The first
// kControlBytes are the control block: status word, then (at +128) the grid
// barrier arrival count and the number of grid barriers completed, and (at
// +1024) the per-token barrier words of a batch's grouped Stage-1 launch; a
// fault clears the whole block.
struct Workspace {
    int* status;        // [0] device status word (0 = ok)
    unsigned* bar;      // grid-barrier arrival count; bar[1] grid barriers completed
    uint32_t* hist;     // [kHistWords] score histogram, zeroed by each call
    float2* part;       // [kMaxSlices][Fp] per-slice proxy partials (g~, u~); a union
                        // batch: its grouped Stage-1 scratch, then its g and u sums
    uint32_t* skey;     // [Fp] every channel's score key (fp32 score bits)
    int* idx_list;      // [Fp] debug: selected channels, ascending
    float* hch;         // [Fp] debug: h per channel (a union batch: the token bits)
    float* dnorm;       // [Fp] ||W_down[:, c]||_2 per channel, written by prepare (persistent)
    uint16_t* x_stage;  // [d] bf16 input staged from host memory (prox_ffn_host)
    float* y_stage;     // [d] fp32 output staged for host memory (prox_ffn_host)
};

size_t workspace_bytes(int d_model, int d_ff);
Workspace carve_workspace(void* base, int d_model, int d_ff);

// ----------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Invalidates an initialised mbarrier.  A step that reuses the shared
// memory of an earlier step in the same launch must invalidate each of its
// mbarriers before initialising it again: re-initialising a valid mbarrier
// is undefined (PTX ISA, mbarrier.init), and on this part such a barrier's
// first phase was never seen to complete by a parity-0 wait.
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Makes mbarrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the given phase parity of an mbarrier, giving up after
// limit_ns or as soon as *abort (when given) becomes non-zero.  Returns
// true when the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long limit_ns, volatile int* abort) {
    // the clock is read only once the phase is clearly late (every 64 polls)
    uint64_t t0 = 0;
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (abort && *abort) return false;
            const uint64_t now = global_timer_ns();
            if (t0 == 0) t0 = now;
            else if ((long long)(now - t0) > limit_ns) return false;
        }
    }
}

// One bulk (TMA, non-tensor) global->shared copy completing on an mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// L2 policy for weights that are read once per call.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ void red_add_v2(float* addr, float a, float b) {
    asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(addr), "f"(a), "f"(b)
                 : "memory");
}

__device__ __forceinline__ void record_status(int* status, int code) {
    atomicCAS(status, 0, code);
}

// ----------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error.  All run on `stream`.
// wq = 0: gateup/down_t receive the bf16 Stage-2 layouts; wq = 1: the int8
// ones (gate|up rows of 2 d + 16 bytes with their scales, W_down^T rows of d
// bytes), see prox_prepare_q8; wq = 2: the int4 ones (d + 16 and d / 2
// bytes), see prox_prepare_q4.
cudaError_t launch_prepare(int d, int F, const __nv_bfloat16* w_gate, const __nv_bfloat16* w_up,
                           const __nv_bfloat16* w_down, uint8_t* codes, __half2* scales,
                           void* gateup, void* down_t, int wq, float* down_norms,
                           cudaStream_t stream);

// Bytes of one Stage-2 gate|up row and one W_down^T row in device memory.
// wq: 0 bf16, 1 int8, 2 int4 (codes, then 16 bytes of row scales).
constexpr size_t gu_row_bytes(int d, int wq) {
    return wq == 2 ? (size_t)d + 16 : wq ? (size_t)2 * d + 16 : (size_t)4 * d;
}
constexpr size_t down_row_bytes(int d, int wq) {
    return wq == 2 ? (size_t)d / 2 : wq ? (size_t)d : (size_t)2 * d;
}

// Proxy work split: `tiles` channel tiles of `tile_w` channels (a multiple
// of 16) times `slices` slices of the kept inputs, tiles * slices <= blocks.
struct ProxyGeom {
    int tiles, slices, tile_w;
};
ProxyGeom proxy_geometry(int F, int kx, int num_blocks, bool any_width = false);

struct FusedLaunch {
    const uint8_t* codes;
    const __half2* scales;
    const void* gateup;  // Stage-2 rows: bf16, int8 or int4 (wq)
    const void* down_t;
    int wq = 0;
    int d, F;
    const uint16_t* x;
    float* y;
    int kx, k;
    int bw = 0;          // block-granular mask: channels per block (0: per channel)
    // second selection signal: rank by |h~_c| ||W_down[:, c]|| (the
    // contribution of channel c) instead of |h~_c|; null: the state signal
    const float* dnorm = nullptr;
    // optional stack glue: x = bf16(RMSNorm(x_prev + y_prev)) computed in the
    // step itself (x unused, x_out receives it); x_prev null: plain step
    const uint16_t* x_prev = nullptr;
    const float* y_prev = nullptr;
    uint16_t* x_out = nullptr;
    float eps = 0.0f;
    // mask only (batch with a union mask): each CTA ORs bit `token` into
    // member[c] for its share of the mask and skips Stage 2 (y is only zeroed)
    uint32_t* member = nullptr;
    int token = 0;
    const Workspace* ws;
    int32_t* kept_out;   // debug outputs, may be null
    float* scores_out;
    int32_t* idx_out;
    float* h_out;
    int num_blocks;
    long long limit_ns;
    int inject;          // test hook: 1 = one CTA withholds the first grid barrier
    uint64_t* ts;        // phase stamps [num_blocks][PROX_PHASE_STAMPS] or null
};

// A stack of layers run in one persistent launch (launch_stack): per layer
// its weights; the layers share shape, workspace and grid.
constexpr int kMaxStack = 64;
struct StackLayer {
    const uint8_t* codes;
    const __half2* scales;
    const uint8_t* gateup;
    const uint8_t* down_t;
};
struct StackLayers {
    int n;
    const uint16_t* x0;  // bf16 [d]: layer 0's input
    uint16_t* xs;        // bf16 [n][d]: x_l for l >= 1 (row 0 unused)
    float* ys;           // fp32 [n][d]: y_l
    StackLayer layer[kMaxStack];
};

cudaError_t fused_configure();
bool fused_fits(int d, int F);
int fused_threads();
int fused_max_chunk();
int fused_max_blocks();
size_t fused_smem_bytes();
cudaError_t launch_fused(const FusedLaunch& L, cudaStream_t stream);
// The stack launch: layers[l] of the same shape (L.wq for all), first
// layer on x0, layer l > 0 on x_l = bf16(RMSNorm(x_{l-1} + y_{l-1}) / eps).
cudaError_t launch_stack(const FusedLaunch& L, const StackLayers& sl, cudaStream_t stream);

// Stage 1 of several tokens in one launch (mask-only steps in groups of
// CTAs): each token's histogram, proxy partials and score keys at
// scratch + t stride (+ part_off, + skey_off); gbar[t] its barrier word
// (zero at launch).  gsize = 0: not possible for this shape and token count.
struct MaskGroupGeom {
    int gsize;
    size_t stride, part_off, skey_off;
};
struct MaskGroups {
    uint8_t* scratch;
    size_t stride, part_off, skey_off;
    unsigned* gbar;
    int token0;  // group t records token bit token0 + t
};
MaskGroupGeom mask_group_geometry(int d, int F, int k, int ntok, int num_blocks);
// L: a mask-only step (member set, bf16 rows, channel mask); L.x / L.y the
// first token's rows, the others follow at d-element strides; their bits
// are token0, token0 + 1, ...
cudaError_t launch_masks(const FusedLaunch& L, int ntok, int token0, uint8_t* scratch,
                         unsigned* gbar, cudaStream_t stream);

// Stage 2 of a batch over the union of its tokens' masks (prox_union.cu):
// G tokens per pass at most (their x staged in shared memory), S gate|up
// ring stages; the W_down^T pass tiles 512-output slices x channel ranges.
constexpr int kUnionMaxG = 8;
struct UnionGeom {
    int G, S, gu_blocks, nslice, nrange, max_items;
    size_t gu_smem, down_smem;
};
UnionGeom union_geometry(int d, int F, int num_blocks);
cudaError_t union_configure();
// GU: [4][G][padded_ff(F)] fp32 scratch (two partial sums each of g and
// u); y: [G][d] fp32, zeroed before (each token's mask-only step zeroes its
// row); member: [F] token bits
cudaError_t launch_union(const void* gateup, const void* down_t, const uint16_t* x,
                         const uint32_t* member, float* GU, float* y, int d, int F, int G,
                         int num_blocks, int* status, long long limit_ns, cudaStream_t stream);
cudaError_t launch_dense(const void* gateup, const void* down_t, int wq, const uint16_t* x, int d,
                         int F, float* y, int* status, int num_blocks, long long limit_ns,
                         uint64_t* ts, cudaStream_t stream);

cudaError_t launch_residual_rmsnorm(int d, const uint16_t* x, const float* y, float eps,
                                    uint16_t* x_next, cudaStream_t stream);

}  // namespace prox

// The host handle behind the opaque prox_layer of prox.h: shapes, grid size
// and the caller's device buffers given to prox_prepare.
struct prox_layer {
    int d_model, d_ff, Fp;
    int device, num_sms, num_blocks;
    const uint8_t* codes;
    const __half2* scales;
    const void* gateup;  // bf16 layouts, or the int8 / int4 ones (wq 1 / 2)
    const void* down_t;
    int wq;
    prox::Workspace ws;
};
