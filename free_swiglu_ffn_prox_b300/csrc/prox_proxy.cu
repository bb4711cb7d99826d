// prox_proxy.cu -- Stage 1 proxy GEMV of "Prox" (Abstract: quantized proxy
// weights applied to the sparsified input approximate the SwiGLU
// intermediate state).  For every channel c:
//     g~_c = sum_g s_gate[c][g] * sum_{j in kept, j/128 = g} q_gate[c][j] x_j
//     u~_c = likewise with the up proxy
// accumulated in fp32 into acc[c] = (g~_c, u~_c); the channel select kernel
// turns them into |silu(g~) u~|.
//
// Work split: the kept rows (one contiguous d_ff-byte row of codes per kept
// input) form a kx x Fp byte matrix.  A CTA takes a 512-channel tile of one
// slice of the kept rows; grid = tiles x slices, sized to fill every SM
// twice in one wave.  Row segments arrive by bulk copies (TMA) into a
// 4-stage ring of 32-row chunks fed by one producer warp; 8 consumer warps
// take the chunk's rows round-robin, each lane owning 16 channels (one
// 16-byte segment of the row).  Per-warp fp32 totals are summed across
// warps in shared memory and added to acc with vector atomics.
//
// Arithmetic per code byte: two offset-binary nibbles become exact fp16
// integers q in [-8, 7] with one LOP3 per two nibbles plus one packed
// HSUB2/HFMA2, then fma.rn.f32.f16 multiplies q by the prescaled fp16 x_j
// and accumulates in fp32 (q * x_j is exact; only the fp32 sums round).
#include "prox_internal.cuh"

namespace prox {
namespace {

constexpr int kTileC = 512;
constexpr int kChunkRows = 32;
constexpr int kStages = 4;
constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (1 + kConsumerWarps);
constexpr int kRedPitch = 33;  // float2 pitch of the cross-warp buffer rows

struct ProxyParams {
    const uint8_t* codes;
    const __half2* scales;
    const uint32_t* kept;
    const int* meta;
    float2* acc;
    int* status;
    int Fp, F, kx, tiles, slices;
    long long limit_ns;
    int inject_stall;
};

struct ProxySmem {
    uint8_t data[kStages][kChunkRows][kTileC];
    uint32_t meta[kStages][kChunkRows];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int last_issued[kStages];
    int abort;
};
static_assert(sizeof(float2) * kConsumerWarps * 16 * kRedPitch <= sizeof(uint8_t) * kStages * kChunkRows * kTileC,
              "cross-warp buffer must fit in the ring");

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

// One 32-bit word = 4 channels (bytes b0..b3, byte = gate | up << 4).
__device__ __forceinline__ void proxy_mac_word(uint32_t w, uint16_t xh, float* ag, float* au) {
    constexpr uint32_t kLo = 0x000F000Fu, kHi = 0x00F000F0u, kMagic = 0x64006400u;
    constexpr uint32_t kBias = 0x64086408u;      // (1032, 1032)
    constexpr uint32_t kSixteenth = 0x2C002C00u; // (1/16, 1/16)
    constexpr uint32_t kHiBias = 0xD480D480u;    // (-72, -72)
    const uint32_t w8 = w >> 8;
    // (1024 + n) and (1024 + 16 n) for the nibbles of bytes 0/2 and 1/3
    const uint32_t g02 = hsub2_bits(lop3_and_or(w, kLo, kMagic), kBias);
    const uint32_t g13 = hsub2_bits(lop3_and_or(w8, kLo, kMagic), kBias);
    const uint32_t u02 = hfma2_bits(lop3_and_or(w, kHi, kMagic), kSixteenth, kHiBias);
    const uint32_t u13 = hfma2_bits(lop3_and_or(w8, kHi, kMagic), kSixteenth, kHiBias);
    fma_f32_f16x2(ag[0], ag[2], g02, xh);
    fma_f32_f16x2(ag[1], ag[3], g13, xh);
    fma_f32_f16x2(au[0], au[2], u02, xh);
    fma_f32_f16x2(au[1], au[3], u13, xh);
}

__global__ void __maxnreg__(112) k_proxy_gemv(const ProxyParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    ProxySmem& sm = *reinterpret_cast<ProxySmem*>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x % p.tiles, slice = blockIdx.x / p.tiles;
    const int c0 = tile * kTileC;
    const int width = min(kTileC, p.Fp - c0);
    const int r0 = (int)((long long)slice * p.kx / p.slices);
    const int r1 = (int)((long long)(slice + 1) * p.kx / p.slices);
    const int nchunks = (r1 - r0 + kChunkRows - 1) / kChunkRows;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerWarps);
            sm.last_issued[s] = -1;
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    float totg[16], totu[16];
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        const uint64_t pol = policy_evict_first();
        for (int i = 0; i < nchunks; ++i) {
            const int s = i % kStages;
            if (i >= kStages) {
                bool ok = true;
                if (lane == 0)
                    ok = mbar_wait_bounded(&sm.empty[s], ((i / kStages) - 1) & 1, p.limit_ns,
                                           &sm.abort);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    if (lane == 0) {
                        sm.abort = 1;
                        record_status(p.status, PROX_ERR_TIMEOUT);
                    }
                    break;
                }
            }
            const int rbeg = r0 + i * kChunkRows;
            const int n = min(kChunkRows, r1 - rbeg);
            uint32_t packed = 0;
            if (lane < n) {
                packed = p.kept[rbeg + lane];
                sm.meta[s][lane] = packed;
            }
            const bool withhold = p.inject_stall && i == 0;  // fault-injection test hook
            __syncwarp();
            if (lane == 0 && !withhold) {
                mbar_arrive_expect_tx(&sm.full[s], (uint32_t)(n * width));
                sm.last_issued[s] = i;
            }
            __syncwarp();
            if (lane < n && !withhold) {
                const uint32_t j = packed >> 16;
                bulk_g2s(&sm.data[s][lane][0], p.codes + (size_t)j * p.Fp + c0, (uint32_t)width,
                         &sm.full[s], pol);
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int cw = warp - 1;
        const bool lane_live = lane * 16 < width;
        float accg[16], accu[16];
        uint4 sc[4];  // 16 (gate, up) fp16 scale pairs of the current group
#pragma unroll
        for (int t = 0; t < 16; ++t) accg[t] = accu[t] = totg[t] = totu[t] = 0.0f;
#pragma unroll
        for (int t = 0; t < 4; ++t) sc[t] = make_uint4(0, 0, 0, 0);
        int cur_g = -1;
        auto flush_pair = [&](uint32_t sv, int c) {
            const float2 s2 = __half22float2(*reinterpret_cast<const __half2*>(&sv));
            totg[c] = fmaf(s2.x, accg[c], totg[c]);
            totu[c] = fmaf(s2.y, accu[c], totu[c]);
            accg[c] = 0.0f;
            accu[c] = 0.0f;
        };
        auto flush = [&]() {
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                flush_pair(sc[t].x, 4 * t + 0);
                flush_pair(sc[t].y, 4 * t + 1);
                flush_pair(sc[t].z, 4 * t + 2);
                flush_pair(sc[t].w, 4 * t + 3);
            }
        };
        for (int i = 0; i < nchunks; ++i) {
            const int s = i % kStages;
            bool ok = true;
            if (lane == 0)
                ok = mbar_wait_bounded(&sm.full[s], (i / kStages) & 1, p.limit_ns, &sm.abort);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    sm.abort = 1;
                    record_status(p.status, PROX_ERR_TIMEOUT);
                }
                break;
            }
            const int n = min(kChunkRows, r1 - (r0 + i * kChunkRows));
            for (int rr = cw; rr < n; rr += kConsumerWarps) {
                const uint32_t packed = sm.meta[s][rr];
                const int g = (int)(packed >> 23);  // j / 128
                if (g != cur_g) {
                    flush();
                    cur_g = g;
                    if (lane_live) {
                        const uint4* src = reinterpret_cast<const uint4*>(
                            p.scales + (size_t)g * p.Fp + c0 + lane * 16);
#pragma unroll
                        for (int t = 0; t < 4; ++t) sc[t] = __ldg(src + t);
                    }
                }
                const uint16_t xh = (uint16_t)(packed & 0xffffu);
                const uint4 w = *reinterpret_cast<const uint4*>(&sm.data[s][rr][lane * 16]);
                proxy_mac_word(w.x, xh, &accg[0], &accu[0]);
                proxy_mac_word(w.y, xh, &accg[4], &accu[4]);
                proxy_mac_word(w.z, xh, &accg[8], &accu[8]);
                proxy_mac_word(w.w, xh, &accg[12], &accu[12]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
        }
        flush();
    }

    __syncthreads();
    if (sm.abort) {
        // drain copies still in flight into this CTA's ring, then leave
        if (threadIdx.x == 0) {
            for (int s = 0; s < kStages; ++s) {
                const int i = sm.last_issued[s];
                if (i >= 0) mbar_wait_bounded(&sm.full[s], (i / kStages) & 1, p.limit_ns, nullptr);
            }
        }
        __syncthreads();
        return;
    }
    // cross-warp sum: red[(cw * 16 + t) * kRedPitch + lane] = (totg[t], totu[t])
    float2* red = reinterpret_cast<float2*>(&sm.data[0][0][0]);
    if (warp > 0) {
        const int cw = warp - 1;
#pragma unroll
        for (int t = 0; t < 16; ++t) red[(cw * 16 + t) * kRedPitch + lane] = make_float2(totg[t], totu[t]);
    }
    __syncthreads();
    const int shift = p.meta[1];
    for (int cl = threadIdx.x; cl < width; cl += kThreads) {
        const int ln = cl >> 4, t = cl & 15;
        float g = 0.0f, u = 0.0f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float2 v = red[(w * 16 + t) * kRedPitch + ln];
            g += v.x;
            u += v.y;
        }
        const int c = c0 + cl;
        if (c < p.F) red_add_v2(&p.acc[c].x, ldexpf(g, -shift), ldexpf(u, -shift));
    }
}

}  // namespace

ProxyGeom proxy_geometry(int F, int kx, int num_sms) {
    const int Fp = padded_ff(F);
    ProxyGeom geo;
    geo.tiles = (Fp + kTileC - 1) / kTileC;
    int slices = (2 * num_sms) / geo.tiles;
    const int max_slices = (kx + 15) / 16;  // at least 16 rows per slice
    if (slices > max_slices) slices = max_slices;
    if (slices < 1) slices = 1;
    geo.slices = slices;
    return geo;
}

cudaError_t proxy_configure() {
    return cudaFuncSetAttribute(k_proxy_gemv, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sizeof(ProxySmem));
}

cudaError_t launch_proxy_gemv(const uint8_t* codes, const __half2* scales, const Workspace& ws,
                              int d, int F, int kx, int num_sms, long long wait_limit_ns,
                              int inject_stall, cudaStream_t stream) {
    (void)d;
    ProxyParams p;
    p.codes = codes;
    p.scales = scales;
    p.kept = ws.kept;
    p.meta = ws.status;
    p.acc = ws.acc;
    p.status = ws.status;
    p.Fp = padded_ff(F);
    p.F = F;
    p.kx = kx;
    const ProxyGeom geo = proxy_geometry(F, kx, num_sms);
    p.tiles = geo.tiles;
    p.slices = geo.slices;
    p.limit_ns = wait_limit_ns;
    p.inject_stall = inject_stall;
    k_proxy_gemv<<<geo.tiles * geo.slices, kThreads, sizeof(ProxySmem), stream>>>(p);
    return cudaGetLastError();
}

}  // namespace prox
