// prox_noalloc.cu -- prox_ffn_noalloc: the decode step with its per-call
// scratch in a fixed array compiled into the library, for callers that can
// not allocate device memory when they run a step.
//
// Who needs it: code that runs under an allocator it does not own (an
// inference server or framework that reserved the whole device up front and
// rejects further cudaMalloc calls), plugins and real-time loops where a
// device allocation would synchronise the device or is forbidden by policy,
// and callers that simply hold the prepared weights but no spare buffer.
// Such callers pass only inputs and outputs; the proxy partials, the score
// histogram, the scores and the grid-barrier words live in `g_scratch`.
//
// The array is a file-scope __device__ variable, so every device that loads
// the library holds kScratchBytes of it until the process exits, and every
// call on a device shares it: calls that overlap on the GPU (two streams,
// two host threads) race on it and must be ordered by the caller.  Host code
// must not pass `g_scratch` itself to a kernel (in host code the name is a
// host-side stand-in, not a device address); the device address is looked up
// once per device with cudaGetSymbolAddress, on the first call made on that
// device, which should therefore come before any stream capture.  The address
// is kept together with the CUDA context it belongs to: after a
// cudaDeviceReset the device's next context loads the library's module again,
// so a call that finds a different current context looks the address up anew
// (again a set-up call, to be made outside any capture).
#include <cuda.h>

#include <mutex>

#include "prox_internal.cuh"

namespace prox {
namespace {

constexpr size_t kScratchBytes = (size_t)4 << 20;  // 4 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
CUcontext g_ctx[kMaxDevices] = {};  // the context each address belongs to

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// The current CUDA context (the driver's cuCtxGetCurrent, reached through
// the runtime, so the library needs no link against the driver library).
cudaError_t current_context(CUcontext* out) {
    static CtxGetCurrentFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e =
            cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p)
            return e != cudaSuccess ? e : cudaErrorNotSupported;
        fn = reinterpret_cast<CtxGetCurrentFn>(p);
    }
    return fn(out) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device address of g_scratch on the current device: set up on the first
// call in each context of the device, then reused.
cudaError_t scratch_address(int dev, void** out) {
    std::lock_guard<std::mutex> lk(g_mu);
    CUcontext ctx = nullptr;
    cudaError_t e = current_context(&ctx);  // null if this thread has no context yet
    if (e != cudaSuccess) return e;
    if (!g_addr[dev] || !ctx || g_ctx[dev] != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);  // makes the primary context current if needed
        if (e == cudaSuccess) e = current_context(&ctx);
        if (e != cudaSuccess) return e;
        g_addr[dev] = p;
        g_ctx[dev] = ctx;
    }
    *out = g_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace prox

extern "C" PROX_API prox_status prox_ffn_noalloc(const prox_layer* layer, const void* x,
                                                 float keep_fraction, float* y,
                                                 prox_stream_t stream) {
    if (!layer || !x || !y) return PROX_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(y) & 15u))
        return PROX_ERR_MISALIGNED;
    const int k = prox_keep_count(layer->d_ff, keep_fraction);
    if (k < 1) return PROX_ERR_INVALID_ARG;
    // the scratch must hold this layer's workspace (proxy partials dominate)
    if (prox::workspace_bytes(layer->d_model, layer->d_ff) > prox::kScratchBytes)
        return PROX_ERR_UNSUPPORTED_SHAPE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return PROX_ERR_CUDA;
    if (dev != layer->device || dev < 0 || dev >= prox::kMaxDevices) return PROX_ERR_INVALID_ARG;
    void* base = nullptr;
    if (prox::scratch_address(dev, &base) != cudaSuccess) return PROX_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents: restart the control block
    // (grid-barrier count, epoch, selection and chunk flags) from zero.  The
    // histogram is cleared by the kernel; everything else is overwritten
    // before it is read.
    if (cudaMemsetAsync(base, 0, prox::kControlBytes, s) != cudaSuccess) return PROX_ERR_CUDA;
    prox::Workspace ws = prox::carve_workspace(base, layer->d_model, layer->d_ff);
    ws.status = layer->ws.status;  // faults stay visible to prox_get_status(layer)
    ws.dnorm = layer->ws.dnorm;    // per-layer data written by prepare
    prox::FusedLaunch f;
    f.codes = layer->codes;
    f.scales = layer->scales;
    f.gateup = layer->gateup;
    f.down_t = layer->down_t;
    f.wq = layer->wq;
    f.d = layer->d_model;
    f.F = layer->d_ff;
    f.x = static_cast<const uint16_t*>(x);
    f.y = y;
    f.kx = prox_keep_count(layer->d_model, 0.5f);
    f.k = k;
    f.ws = &ws;
    f.kept_out = nullptr;
    f.scores_out = nullptr;
    f.idx_out = nullptr;
    f.h_out = nullptr;
    f.num_blocks = layer->num_blocks;
    f.limit_ns = prox::kWaitLimitNs;
    f.inject = 0;
    f.ts = nullptr;
    return prox::launch_fused(f, s) == cudaSuccess ? PROX_OK : PROX_ERR_CUDA;
}
