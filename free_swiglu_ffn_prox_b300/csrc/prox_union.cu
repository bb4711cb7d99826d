// Stage 2 of a batch of decode tokens over the union of their channel masks.
//
// Every token keeps its own exact mask (Prox, Abstract: one channel mask per
// token, from the magnitude ranking of its proxy state) and its own output:
// y_t = sum over c in mask_t of W_down[:, c] silu(g_t,c) u_t,c, the SwiGLU
// block of PrunePath Sec. 2.1 Eq. (1) restricted to mask_t.  Only the reads
// are shared: each row in the union of the masks streams from HBM once and
// serves every token whose mask holds it.
//
//   member[c]      bit t set when token t's mask holds channel c (each
//                  token's mask-only step ORs its bit in);
//   k_union_gu     CTA b takes the union channels of [F b / n, F (b + 1) / n).
//                  One producer lane streams their gate|up rows by bulk
//                  copies into a ring of S stages.  Two consumer warps share
//                  each stage, each taking every other 8-element chunk of the
//                  row: for each token t holding the channel a warp forms its
//                  part of g = W_gate[c] . x_t and u = W_up[c] . x_t in fp32
//                  (packed pairs of FMAs) and writes the two partial sums to
//                  GU[part][t][c] (no synchronisation between the warps).
//   k_union_down   CTA (s, r) takes the 512-output slice s of the W_down^T
//                  rows of the union channels in range r.  When it stages the
//                  range's items it forms h = silu(g) u from the two parts'
//                  sums (0 where a token's mask lacks c).  Each thread owns 8
//                  outputs of the slice in one of 8 row groups, streams its
//                  16-byte pieces of the rows through a cp.async ring and
//                  accumulates y_t += h_t,c W_down^T[c, slice] for all 8
//                  token slots, two outputs per packed FMA.  The row groups
//                  are summed in shared memory and added to y with one vector
//                  reduction per 4 outputs and token.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "prox_internal.cuh"

namespace prox {
namespace {

constexpr int kUMaxStages = 9;
constexpr int kParts = 2;                // consumer warps per gate|up stage
constexpr int kUItems = 256;             // union channels per k_union_gu CTA at most
constexpr int kDownThreads = 512;        // k_union_down: 8 row groups x 64 threads
constexpr int kDownGroups = 8;
constexpr int kDownSlice = 512;          // outputs per k_union_down CTA (8 per thread)
constexpr int kDownRing = 12;            // 16-byte pieces in flight per thread
constexpr size_t kUnionSmem = 226 * 1024;  // dynamic, under the 227 KB a CTA may opt in to

struct UCtl {
    uint64_t full[kUMaxStages], empty[kUMaxStages];
    int last[kUMaxStages];
    int n;
    int abort;
};
constexpr size_t ctl_span() { return (sizeof(UCtl) + 127) / 128 * 128; }

struct UnionGuArgs {
    const uint8_t* gateup;   // [F] rows of 4 d bytes: bf16 W_gate[c] then W_up[c]
    const uint16_t* x;       // [G][d] bf16
    const uint32_t* member;  // [F]
    float* GU;               // [2][kParts][G][Fp]: partial g sums, then partial u sums
    int d, F, Fp, G, S;
    int* status;
    long long limit_ns;
};

// the 8 bf16 of a 16-byte word as 4 pairs (elements 2e, 2e + 1)
__device__ __forceinline__ void unpack8x2(const uint4 v, float2* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) f[e] = make_float2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xffff0000u));
}

// Waits for a phase (every lane polls); on a timeout records the status and
// raises the CTA's abort flag.
__device__ __forceinline__ bool uwait(uint64_t* bar, uint32_t parity, UCtl& ctl, int* status,
                                      long long limit_ns) {
    const bool got = mbar_wait_bounded(bar, parity, limit_ns, &ctl.abort);
    if (!got) {
        ctl.abort = 1;
        record_status(status, PROX_ERR_TIMEOUT);
    }
    return got;
}

__global__ void __launch_bounds__(32 * (1 + kParts * kUMaxStages), 1) k_union_gu(const UnionGuArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    UCtl& ctl = *reinterpret_cast<UCtl*>(smem);
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + ctl_span());            // [G][d]
    int* item = reinterpret_cast<int*>(xs + (size_t)a.G * a.d);                // [kUItems]
    uint32_t* bits = reinterpret_cast<uint32_t*>(item + kUItems);              // [kUItems]
    uint8_t* ring = reinterpret_cast<uint8_t*>(bits + kUItems);                // [S][4 d]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d, S = a.S, nchunk = d / 8;
    const uint32_t rb = (uint32_t)(4 * d);
    const int c0 = (int)((long long)a.F * blockIdx.x / gridDim.x);
    const int c1 = (int)((long long)a.F * (blockIdx.x + 1) / gridDim.x);  // c1 - c0 <= kUItems (host)

    const int nx = a.G * nchunk;
    for (int i = tid; i < nx; i += blockDim.x)
        reinterpret_cast<uint4*>(xs)[i] = __ldg(reinterpret_cast<const uint4*>(a.x) + i);
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&ctl.full[s], 1);
            mbar_init(&ctl.empty[s], kParts);  // both warps of the stage are done with it
            ctl.last[s] = -1;
        }
        ctl.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {  // the range's union channels, ascending
        int n = 0;
        for (int base = c0; base < c1; base += 32) {
            const int c = base + lane;
            const uint32_t m = c < c1 ? __ldg(a.member + c) : 0u;
            const unsigned bal = __ballot_sync(0xffffffffu, m != 0u);
            if (m) {
                const int pos = n + __popc(bal & ((1u << lane) - 1u));
                item[pos] = c;
                bits[pos] = m;
            }
            n += __popc(bal);
        }
        if (lane == 0) ctl.n = n;
    }
    __syncthreads();
    const int n = ctl.n;

    if (warp == 0) {
        if (lane == 0) {  // producer
            const uint64_t pol = policy_evict_first();
            for (int i = 0; i < n; ++i) {
                const int s = i % S;
                if (i >= S && !uwait(&ctl.empty[s], (uint32_t)((i / S) - 1) & 1u, ctl, a.status,
                                     a.limit_ns))
                    break;
                if (*reinterpret_cast<volatile int*>(&ctl.abort)) break;
                ctl.last[s] = i;
                mbar_arrive_expect_tx(&ctl.full[s], rb);
                bulk_g2s(ring + (size_t)s * rb, a.gateup + (size_t)item[i] * rb, rb, &ctl.full[s], pol);
            }
        }
    } else if (warp <= kParts * S) {
        const int s = (warp - 1) % S, part = (warp - 1) / S;
        const uint4* xv = reinterpret_cast<const uint4*>(xs);
        const uint4* gr = reinterpret_cast<const uint4*>(ring + (size_t)s * rb);
        const uint4* ur = gr + nchunk;
        float* gsum = a.GU + (size_t)part * a.G * a.Fp;
        float* usum = a.GU + (size_t)(kParts + part) * a.G * a.Fp;
        for (int i = s; i < n; i += S) {
            const bool got = mbar_wait_bounded(&ctl.full[s], (uint32_t)(i / S) & 1u, a.limit_ns,
                                               &ctl.abort);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) {
                    ctl.abort = 1;
                    record_status(a.status, PROX_ERR_TIMEOUT);
                }
                break;
            }
            const uint32_t m = bits[i];
            float2 g[kUnionMaxG], u[kUnionMaxG];  // even / odd element partial sums
#pragma unroll
            for (int t = 0; t < kUnionMaxG; ++t) g[t] = u[t] = make_float2(0.0f, 0.0f);
            for (int ch = lane + 32 * part; ch < nchunk; ch += 32 * kParts) {
                float2 gf[4], uf[4];
                unpack8x2(gr[ch], gf);
                unpack8x2(ur[ch], uf);
#pragma unroll
                for (int t = 0; t < kUnionMaxG; ++t)
                    if ((m >> t) & 1u) {
                        float2 xf[4];
                        unpack8x2(xv[(size_t)t * nchunk + ch], xf);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            g[t] = __ffma2_rn(gf[e], xf[e], g[t]);
                            u[t] = __ffma2_rn(uf[e], xf[e], u[t]);
                        }
                    }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.empty[s]);  // every lane is done with the stage
            const int c = item[i];
#pragma unroll
            for (int t = 0; t < kUnionMaxG; ++t)
                if ((m >> t) & 1u) {
                    float gt = g[t].x + g[t].y, ut = u[t].x + u[t].y;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        gt += __shfl_xor_sync(0xffffffffu, gt, o);
                        ut += __shfl_xor_sync(0xffffffffu, ut, o);
                    }
                    if (lane == 0) {
                        gsum[(size_t)t * a.Fp + c] = gt;
                        usum[(size_t)t * a.Fp + c] = ut;
                    }
                }
        }
    }
    __syncthreads();
    // after an abort, the copies still in flight land before the CTA leaves
    if (tid == 0 && ctl.abort)
        for (int s = 0; s < S; ++s)
            if (ctl.last[s] >= 0)
                mbar_wait_bounded(&ctl.full[s], (uint32_t)(ctl.last[s] / S) & 1u, a.limit_ns, nullptr);
}

struct UnionDownArgs {
    const uint8_t* down_t;   // [F] rows of 2 d bytes (bf16 W_down^T[c])
    const uint32_t* member;  // [F]
    const float* GU;         // [2][kParts][G][Fp] partial g and u sums
    float* y;                // [G][d], accumulated into
    int d, F, Fp, G, nslice, nrange, max_items;
};

__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(kDownThreads, 1) k_union_down(const UnionDownArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    // ring [kDownRing][kDownThreads] uint4, later the row-group sums
    // [4][kUnionMaxG][kDownSlice] float (64 KB of its 96 KB); then the items,
    // their member bits and their h values [max_items][kUnionMaxG]
    uint4* ring = reinterpret_cast<uint4*>(smem);
    float* red = reinterpret_cast<float*>(smem);
    int* item = reinterpret_cast<int*>(smem + (size_t)kDownRing * kDownThreads * 16);
    uint32_t* bits = reinterpret_cast<uint32_t*>(item + a.max_items);
    float* hs = reinterpret_cast<float*>(bits + a.max_items);  // 16-byte aligned: max_items % 4 == 0
    __shared__ int wcount[kDownThreads / 32], n_items;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.G, d = a.d;
    const int sl = blockIdx.x % a.nslice, r = blockIdx.x / a.nslice;
    const int e0 = sl * kDownSlice, width = min(kDownSlice, d - e0);
    const int c0 = (int)((long long)a.F * r / a.nrange), c1 = (int)((long long)a.F * (r + 1) / a.nrange);

    // the range's union channels, ascending: each warp counts a contiguous
    // part, then writes it after the warps before it
    const int len = c1 - c0, per = (len + kDownThreads / 32 - 1) / (kDownThreads / 32);
    const int w0 = c0 + min(len, warp * per), w1 = c0 + min(len, (warp + 1) * per);
    int cnt = 0;
    for (int base = w0; base < w1; base += 32) {
        const int c = base + lane;
        cnt += __popc(__ballot_sync(0xffffffffu, c < w1 && __ldg(a.member + c) != 0u));
    }
    if (lane == 0) wcount[warp] = cnt;
    __syncthreads();
    int pos = 0;
    for (int w = 0; w < warp; ++w) pos += wcount[w];
    if (warp == kDownThreads / 32 - 1 && lane == 0) n_items = pos + cnt;
    for (int base = w0; base < w1; base += 32) {
        const int c = base + lane;
        const uint32_t m = c < w1 ? __ldg(a.member + c) : 0u;
        const unsigned bal = __ballot_sync(0xffffffffu, m != 0u);
        if (m) {
            const int p = pos + __popc(bal & ((1u << lane) - 1u));
            item[p] = c;
            bits[p] = m;
        }
        pos += __popc(bal);
    }
    __syncthreads();
    const int n = n_items;  // <= max_items (host: c1 - c0 <= max_items)
    for (int q = tid; q < n * kUnionMaxG; q += kDownThreads) {
        const int i = q / kUnionMaxG, t = q % kUnionMaxG;
        float h = 0.0f;
        if (t < G && ((bits[i] >> t) & 1u)) {
            float g = 0.0f, u = 0.0f;
#pragma unroll
            for (int p = 0; p < kParts; ++p) {
                g += __ldg(a.GU + ((size_t)p * G + t) * a.Fp + item[i]);
                u += __ldg(a.GU + ((size_t)(kParts + p) * G + t) * a.Fp + item[i]);
            }
            h = g / (1.0f + expf(-g)) * u;  // silu(g) u
        }
        hs[q] = h;
    }
    __syncthreads();

    constexpr int kTpr = kDownSlice / 8;  // threads per row slice
    const int rg = tid / kTpr, cp = tid % kTpr;
    const bool act = 8 * cp < width;
    float2 acc[kUnionMaxG][4];
#pragma unroll
    for (int t = 0; t < kUnionMaxG; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[t][e] = make_float2(0.0f, 0.0f);
    const size_t rowb = (size_t)2 * d;
    const uint8_t* col = a.down_t + (size_t)(e0 + 8 * cp) * 2;
    uint4* my = ring + tid;
    if (act) {
#pragma unroll
        for (int u = 0; u < kDownRing; ++u) {
            const int q = rg + kDownGroups * u;
            if (q < n) cp_async_16(my + (size_t)u * kDownThreads, col + (size_t)item[q] * rowb);
            cp_commit();
        }
        int s = 0;
#pragma unroll 1
        for (int i = rg; i < n; i += kDownGroups) {
            cp_wait<kDownRing - 1>();
            const uint4 w = my[(size_t)s * kDownThreads];
            const int qn = i + kDownGroups * kDownRing;
            if (qn < n) cp_async_16(my + (size_t)s * kDownThreads, col + (size_t)item[qn] * rowb);
            cp_commit();
            s = s + 1 == kDownRing ? 0 : s + 1;
            float2 wf[4];
            unpack8x2(w, wf);
            const float4 h0 = *reinterpret_cast<const float4*>(hs + (size_t)i * kUnionMaxG);
            const float4 h1 = *reinterpret_cast<const float4*>(hs + (size_t)i * kUnionMaxG + 4);
            const float hv[kUnionMaxG] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
            for (int t = 0; t < kUnionMaxG; ++t) {
                const float2 h2 = make_float2(hv[t], hv[t]);
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[t][e] = __ffma2_rn(h2, wf[e], acc[t][e]);
            }
        }
        cp_wait<0>();
    }
    __syncthreads();  // the ring becomes the row-group sums
    // two rounds: groups 4..7 store, then groups 0..3 add theirs in place
    auto slot = [&](int g, int t) { return red + ((size_t)g * kUnionMaxG + t) * kDownSlice + 8 * cp; };
    if (act && rg >= kDownGroups / 2)
#pragma unroll
        for (int t = 0; t < kUnionMaxG; ++t) {
            float4* dst = reinterpret_cast<float4*>(slot(rg - kDownGroups / 2, t));
            dst[0] = make_float4(acc[t][0].x, acc[t][0].y, acc[t][1].x, acc[t][1].y);
            dst[1] = make_float4(acc[t][2].x, acc[t][2].y, acc[t][3].x, acc[t][3].y);
        }
    __syncthreads();
    if (act && rg < kDownGroups / 2)
#pragma unroll
        for (int t = 0; t < kUnionMaxG; ++t) {
            float4* dst = reinterpret_cast<float4*>(slot(rg, t));
            float4 p0 = dst[0], p1 = dst[1];
            p0.x += acc[t][0].x; p0.y += acc[t][0].y; p0.z += acc[t][1].x; p0.w += acc[t][1].y;
            p1.x += acc[t][2].x; p1.y += acc[t][2].y; p1.z += acc[t][3].x; p1.w += acc[t][3].y;
            dst[0] = p0;
            dst[1] = p1;
        }
    __syncthreads();
    if (n == 0) return;
    for (int q = tid; q < G * (kDownSlice / 4); q += kDownThreads) {
        const int t = q / (kDownSlice / 4), c4 = q % (kDownSlice / 4);
        if (4 * c4 >= width) continue;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int g = 0; g < kDownGroups / 2; ++g) {
            const float4 p = *reinterpret_cast<const float4*>(red + ((size_t)g * kUnionMaxG + t) * kDownSlice + 4 * c4);
            v.x += p.x;
            v.y += p.y;
            v.z += p.z;
            v.w += p.w;
        }
        red_add_v4(a.y + (size_t)t * d + e0 + 4 * c4, v.x, v.y, v.z, v.w);
    }
}

}  // namespace

UnionGeom union_geometry(int d, int F, int num_blocks) {
    UnionGeom g{};
    // gate|up: G tokens' x (2 d bytes each) and S >= 3 ring stages of 4 d
    // bytes next to the control block and the item list
    const size_t fixed = ctl_span() + (size_t)kUItems * 8;
    for (int G = kUnionMaxG; G >= 1; --G) {
        const size_t left = kUnionSmem > fixed + (size_t)G * 2 * d ? kUnionSmem - fixed - (size_t)G * 2 * d : 0;
        const int S = (int)std::min<size_t>(kUMaxStages, left / ((size_t)4 * d));
        if (S >= 3) {
            g.G = G;
            g.S = S;
            break;
        }
    }
    g.gu_blocks = std::max(num_blocks, (F + kUItems - 1) / kUItems);
    g.gu_smem = fixed + (size_t)g.G * 2 * d + (size_t)g.S * 4 * d;
    // down: slices of 512 outputs x channel ranges, about one CTA per SM;
    // a range's items, bits and h values fit next to the 96 KB ring
    g.nslice = (d + kDownSlice - 1) / kDownSlice;
    const size_t ring = (size_t)kDownRing * kDownThreads * 16;
    const size_t per_item = 8 + (size_t)4 * kUnionMaxG;
    const int max_range = (int)((kUnionSmem - ring) / per_item) - 4;
    g.nrange = std::max(std::max(1, num_blocks / g.nslice), (F + max_range - 1) / max_range);
    g.max_items = ((F + g.nrange - 1) / g.nrange + 4) / 4 * 4;
    g.down_smem = ring + (size_t)g.max_items * per_item;
    return g;
}

cudaError_t union_configure() {
    cudaError_t e = cudaFuncSetAttribute(k_union_gu, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kUnionSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_union_down, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kUnionSmem);
    return e;
}

cudaError_t launch_union(const void* gateup, const void* down_t, const uint16_t* x,
                         const uint32_t* member, float* GU, float* y, int d, int F, int G,
                         int num_blocks, int* status, long long limit_ns, cudaStream_t stream) {
    const UnionGeom g = union_geometry(d, F, num_blocks);
    if (G < 1 || G > g.G) return cudaErrorInvalidValue;
    UnionGuArgs a;
    a.gateup = static_cast<const uint8_t*>(gateup);
    a.x = x;
    a.member = member;
    a.GU = GU;
    a.d = d;
    a.F = F;
    a.Fp = padded_ff(F);
    a.G = G;
    a.S = g.S;
    a.status = status;
    a.limit_ns = limit_ns;
    const size_t smem_a = ctl_span() + (size_t)kUItems * 8 + (size_t)G * 2 * d + (size_t)g.S * 4 * d;
    k_union_gu<<<g.gu_blocks, 32 * (1 + kParts * g.S), smem_a, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    UnionDownArgs b;
    b.down_t = static_cast<const uint8_t*>(down_t);
    b.member = member;
    b.GU = GU;
    b.y = y;
    b.d = d;
    b.F = F;
    b.Fp = padded_ff(F);
    b.G = G;
    b.nslice = g.nslice;
    b.nrange = g.nrange;
    b.max_items = g.max_items;
    const size_t smem_b = (size_t)kDownRing * kDownThreads * 16 + (size_t)g.max_items * (8 + (size_t)4 * kUnionMaxG);
    k_union_down<<<g.nslice * g.nrange, kDownThreads, smem_b, stream>>>(b);
    return cudaGetLastError();
}

}  // namespace prox
