// prox_abi.cu -- the extern "C" entry points declared in include/prox.h:
// argument checks, workspace carving, and the launch of the Prox decode step
// ("Prox", Abstract), which runs as one persistent kernel (prox_fused.cu):
// input sparsity, proxy GEMV, channel mask and exact Stage 2.
#include <math.h>
#include <stdlib.h>

#include <new>

#include <algorithm>

#include "prox_internal.cuh"

namespace prox {

static size_t align256(size_t v) { return (v + 255) / 256 * 256; }

size_t workspace_bytes(int d, int F) {
    const size_t Fp = (size_t)padded_ff(F);
    return kControlBytes + align256((size_t)kHistWords * 4) +
           align256((size_t)kMaxSlices * Fp * 8) + 4 * align256(Fp * 4) +
           align256((size_t)d * 2) + align256((size_t)d * 4);
}

Workspace carve_workspace(void* base, int d, int F) {
    const size_t Fp = (size_t)padded_ff(F);
    uint8_t* p = static_cast<uint8_t*>(base);
    Workspace w;
    w.status = reinterpret_cast<int*>(p);
    w.bar = reinterpret_cast<unsigned*>(p + 128);
    p += kControlBytes;
    w.hist = reinterpret_cast<uint32_t*>(p);
    p += align256((size_t)kHistWords * 4);
    w.part = reinterpret_cast<float2*>(p);
    p += align256((size_t)kMaxSlices * Fp * 8);
    w.skey = reinterpret_cast<uint32_t*>(p);
    p += align256(Fp * 4);
    w.idx_list = reinterpret_cast<int*>(p);
    p += align256(Fp * 4);
    w.hch = reinterpret_cast<float*>(p);
    p += align256(Fp * 4);
    w.dnorm = reinterpret_cast<float*>(p);
    p += align256(Fp * 4);
    w.x_stage = reinterpret_cast<uint16_t*>(p);
    p += align256((size_t)d * 2);
    w.y_stage = reinterpret_cast<float*>(p);
    return w;
}

}  // namespace prox

namespace {

bool shape_ok(int d, int F) {
    return d >= prox::kGroup && d <= prox::kMaxDModel && d % prox::kGroup == 0 && F >= 1 &&
           F <= prox::kMaxDff && prox::fused_fits(d, F);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool frac_ok(float f) { return isfinite(f) && f > 0.0f && f <= 1.0f; }

prox_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PROX_OK : PROX_ERR_CUDA; }

// Records `ev` on the stream; inside a stream capture it becomes an event
// node of the graph, so traced calls can be captured too.
cudaError_t record(cudaEvent_t ev, cudaStream_t stream) {
    if (!ev) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) return e;
    return cs == cudaStreamCaptureStatusActive
               ? cudaEventRecordWithFlags(ev, stream, cudaEventRecordExternal)
               : cudaEventRecord(ev, stream);
}

// The decode step on a checked layer.  kept_out/scores_out/idx_out/h_out
// are the debug outputs (NULL on the hot path); ev (NULL or
// PROX_TRACE_EVENTS events) brackets the kernel.
prox_status run_prox(const prox_layer* L, const void* x, float keep_fraction, float input_keep,
                     float* y, int32_t* kept_out, float* scores_out, int32_t* idx_out,
                     float* h_out, cudaStream_t stream, long long limit_ns, int inject,
                     cudaEvent_t const* ev = nullptr, uint64_t* ts = nullptr,
                     const void* x_prev = nullptr, const float* y_prev = nullptr,
                     void* x_out = nullptr, float eps = 0.0f, int bw = 0,
                     bool contrib = false) {
    prox::FusedLaunch f;
    f.codes = L->codes;
    f.scales = L->scales;
    f.gateup = L->gateup;
    f.down_t = L->down_t;
    f.wq = L->wq;
    f.d = L->d_model;
    f.F = L->d_ff;
    f.x = static_cast<const uint16_t*>(x);
    f.y = y;
    f.kx = prox_keep_count(L->d_model, input_keep);
    f.k = bw > 0 ? bw * prox_keep_count(L->d_ff / bw, keep_fraction)  // whole blocks
                 : prox_keep_count(L->d_ff, keep_fraction);
    f.bw = bw;
    f.dnorm = contrib ? L->ws.dnorm : nullptr;
    f.ws = &L->ws;
    f.kept_out = kept_out;
    f.scores_out = scores_out;
    f.idx_out = idx_out;
    f.h_out = h_out;
    f.num_blocks = L->num_blocks;
    f.limit_ns = limit_ns;
    f.inject = inject;
    f.ts = ts;
    f.x_prev = static_cast<const uint16_t*>(x_prev);
    f.y_prev = y_prev;
    f.x_out = static_cast<uint16_t*>(x_out);
    f.eps = eps;
    cudaError_t e = ev ? record(ev[0], stream) : cudaSuccess;
    if (e == cudaSuccess) e = prox::launch_fused(f, stream);
    if (e == cudaSuccess && ev) e = record(ev[1], stream);
    return cuda_status(e);
}

// Whether the byte ranges [a, a + na) and [b, b + nb) overlap.
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

// A block width the fused kernel supports on this layer: a power of two in
// [4, 256] dividing d_ff, at least one block per CTA, and every CTA's chunk
// (whole blocks) within the kernel's chunk limit.
prox_status check_blocks(const prox_layer* L, int bw) {
    if (bw < 4 || bw > 256 || (bw & (bw - 1)) != 0) return PROX_ERR_INVALID_ARG;
    if (L->d_ff % bw != 0) return PROX_ERR_UNSUPPORTED_SHAPE;
    const int E = L->d_ff / bw, nb = L->num_blocks;
    if (E < nb || bw * ((E + nb - 1) / nb) > prox::fused_max_chunk())
        return PROX_ERR_UNSUPPORTED_SHAPE;
    return PROX_OK;
}

prox_status check_call(const prox_layer* L, const void* x, const float* y) {
    if (!L || !x || !y) return PROX_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return PROX_ERR_MISALIGNED;
    return PROX_OK;
}

prox_status query_sizes(int d_model, int d_ff, int wq, prox_sizes* out) {
    if (!out) return PROX_ERR_INVALID_ARG;
    if (!shape_ok(d_model, d_ff)) return PROX_ERR_UNSUPPORTED_SHAPE;
    const size_t Fp = (size_t)prox::padded_ff(d_ff);
    out->proxy_codes = (size_t)d_model * Fp;
    out->proxy_scales = (size_t)(d_model / prox::kGroup) * Fp * 4;
    out->gateup = (size_t)d_ff * prox::gu_row_bytes(d_model, wq);
    out->down_t = (size_t)d_ff * prox::down_row_bytes(d_model, wq);
    out->workspace = prox::workspace_bytes(d_model, d_ff);
    return PROX_OK;
}

prox_status prepare(int d_model, int d_ff, const void* w_gate, const void* w_up,
                    const void* w_down, void* proxy_codes, void* proxy_scales, void* gateup,
                    void* down_t, void* workspace, prox_stream_t stream, int wq,
                    prox_layer** out) {
    if (!out) return PROX_ERR_INVALID_ARG;
    *out = nullptr;
    if (!shape_ok(d_model, d_ff)) return PROX_ERR_UNSUPPORTED_SHAPE;
    const void* ptrs[] = {w_gate, w_up, w_down, proxy_codes, proxy_scales, gateup, down_t, workspace};
    for (const void* p : ptrs) {
        if (!p) return PROX_ERR_INVALID_ARG;
        if (!aligned16(p)) return PROX_ERR_MISALIGNED;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = prox::fused_configure();
    if (e == cudaSuccess) e = prox::union_configure();
    if (e == cudaSuccess)
        e = cudaMemsetAsync(workspace, 0, prox::workspace_bytes(d_model, d_ff), s);
    if (e == cudaSuccess)
        e = prox::launch_prepare(d_model, d_ff, static_cast<const __nv_bfloat16*>(w_gate),
                                 static_cast<const __nv_bfloat16*>(w_up),
                                 static_cast<const __nv_bfloat16*>(w_down),
                                 static_cast<uint8_t*>(proxy_codes),
                                 static_cast<__half2*>(proxy_scales),
                                 gateup, down_t, wq,
                                 prox::carve_workspace(workspace, d_model, d_ff).dnorm, s);
    if (e != cudaSuccess) return PROX_ERR_CUDA;
    // one persistent CTA per SM; every CTA holds its chunk of the channels
    // in shared memory
    const int g4 = (d_ff + 3) / 4;  // chunks start on multiples of 4 channels
    if (sms > prox::fused_max_blocks() || 4 * ((g4 + sms - 1) / sms) > prox::fused_max_chunk())
        return PROX_ERR_UNSUPPORTED_SHAPE;
    prox_layer* L = new (std::nothrow) prox_layer;
    if (!L) return PROX_ERR_INVALID_ARG;
    L->d_model = d_model;
    L->d_ff = d_ff;
    L->Fp = prox::padded_ff(d_ff);
    L->device = dev;
    L->num_sms = sms;
    L->num_blocks = sms;
    L->codes = static_cast<const uint8_t*>(proxy_codes);
    L->scales = static_cast<const __half2*>(proxy_scales);
    L->gateup = gateup;
    L->down_t = down_t;
    L->wq = wq;
    L->ws = prox::carve_workspace(workspace, d_model, d_ff);
    *out = L;
    return PROX_OK;
}

}  // namespace

extern "C" {

int prox_keep_count(int n, float frac) {
    if (n < 1 || !frac_ok(frac)) return 0;
    double k = ceil((double)frac * (double)n);
    if (k < 1.0) k = 1.0;
    if (k > (double)n) k = (double)n;
    return (int)k;
}

const char* prox_status_string(prox_status s) {
    switch (s) {
        case PROX_OK: return "ok";
        case PROX_ERR_INVALID_ARG: return "invalid argument";
        case PROX_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case PROX_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
        case PROX_ERR_CUDA: return "CUDA runtime error";
        case PROX_ERR_TIMEOUT: return "bounded device wait ran out";
        case PROX_ERR_DEVICE_CHECK: return "device-side check failed";
    }
    return "unknown status";
}

prox_status prox_query_sizes(int d_model, int d_ff, prox_sizes* out) {
    return query_sizes(d_model, d_ff, 0, out);
}

prox_status prox_query_sizes_q8(int d_model, int d_ff, prox_sizes* out) {
    return query_sizes(d_model, d_ff, 1, out);
}

prox_status prox_query_sizes_q4(int d_model, int d_ff, prox_sizes* out) {
    return query_sizes(d_model, d_ff, 2, out);
}

prox_status prox_prepare(int d_model, int d_ff, const void* w_gate, const void* w_up,
                         const void* w_down, void* proxy_codes, void* proxy_scales,
                         void* gateup, void* down_t, void* workspace, prox_stream_t stream,
                         prox_layer** out) {
    return prepare(d_model, d_ff, w_gate, w_up, w_down, proxy_codes, proxy_scales, gateup, down_t,
                   workspace, stream, 0, out);
}

prox_status prox_prepare_q8(int d_model, int d_ff, const void* w_gate, const void* w_up,
                            const void* w_down, void* proxy_codes, void* proxy_scales,
                            void* gateup_q8, void* down_q8, void* workspace, prox_stream_t stream,
                            prox_layer** out) {
    return prepare(d_model, d_ff, w_gate, w_up, w_down, proxy_codes, proxy_scales, gateup_q8,
                   down_q8, workspace, stream, 1, out);
}

prox_status prox_prepare_q4(int d_model, int d_ff, const void* w_gate, const void* w_up,
                            const void* w_down, void* proxy_codes, void* proxy_scales,
                            void* gateup_q4, void* down_q4, void* workspace, prox_stream_t stream,
                            prox_layer** out) {
    return prepare(d_model, d_ff, w_gate, w_up, w_down, proxy_codes, proxy_scales, gateup_q4,
                   down_q4, workspace, stream, 2, out);
}

prox_status prox_ffn_ex(const prox_layer* layer, const void* x, float keep_fraction,
                        float input_keep, float* y, prox_stream_t stream) {
    prox_status st = check_call(layer, x, y);
    if (st != PROX_OK) return st;
    if (!frac_ok(keep_fraction) || !frac_ok(input_keep)) return PROX_ERR_INVALID_ARG;
    return run_prox(layer, x, keep_fraction, input_keep, y, nullptr, nullptr, nullptr, nullptr,
                    reinterpret_cast<cudaStream_t>(stream), prox::kWaitLimitNs, 0);
}

prox_status prox_ffn(const prox_layer* layer, const void* x, float keep_fraction, float* y,
                     prox_stream_t stream) {
    return prox_ffn_ex(layer, x, keep_fraction, 0.5f, y, stream);
}

prox_status prox_ffn_host(const prox_layer* layer, const void* x_host, float keep_fraction,
                          float* y_host, prox_stream_t stream) {
    if (!layer || !x_host || !y_host) return PROX_ERR_INVALID_ARG;
    if (!frac_ok(keep_fraction)) return PROX_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int d = layer->d_model;
    cudaError_t e = cudaMemcpyAsync(layer->ws.x_stage, x_host, (size_t)d * 2,
                                    cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return PROX_ERR_CUDA;
    prox_status st = run_prox(layer, layer->ws.x_stage, keep_fraction, 0.5f, layer->ws.y_stage,
                              nullptr, nullptr, nullptr, nullptr, s, prox::kWaitLimitNs, 0);
    if (st != PROX_OK) return st;
    e = cudaMemcpyAsync(y_host, layer->ws.y_stage, (size_t)d * 4, cudaMemcpyDeviceToHost, s);
    return cuda_status(e);
}

prox_status prox_ffn_traced(const prox_layer* layer, const void* x, float keep_fraction,
                            float input_keep, float* y, void* const* events, int n_events,
                            prox_stream_t stream) {
    prox_status st = check_call(layer, x, y);
    if (st != PROX_OK) return st;
    if (!frac_ok(keep_fraction) || !frac_ok(input_keep)) return PROX_ERR_INVALID_ARG;
    if (!events || n_events != PROX_TRACE_EVENTS) return PROX_ERR_INVALID_ARG;
    for (int i = 0; i < n_events; ++i)
        if (!events[i]) return PROX_ERR_INVALID_ARG;
    return run_prox(layer, x, keep_fraction, input_keep, y, nullptr, nullptr, nullptr, nullptr,
                    reinterpret_cast<cudaStream_t>(stream), prox::kWaitLimitNs, 0,
                    reinterpret_cast<cudaEvent_t const*>(events));
}

prox_status prox_ffn_resnorm(const prox_layer* layer, const void* x_prev, const float* y_prev,
                             float eps, void* x_out, float keep_fraction, float* y,
                             prox_stream_t stream) {
    if (!layer || !x_prev || !y_prev || !x_out || !y) return PROX_ERR_INVALID_ARG;
    if (!aligned16(x_prev) || !aligned16(y_prev) || !aligned16(x_out) || !aligned16(y))
        return PROX_ERR_MISALIGNED;
    if (!frac_ok(keep_fraction) || !(eps >= 0.0f) || !isfinite(eps)) return PROX_ERR_INVALID_ARG;
    const size_t d = (size_t)layer->d_model;
    // every CTA reads x_prev and y_prev while CTA 0 writes x_out and clears y
    if (overlap(x_out, 2 * d, x_prev, 2 * d) || overlap(x_out, 2 * d, y_prev, 4 * d) ||
        overlap(x_out, 2 * d, y, 4 * d) || overlap(y, 4 * d, y_prev, 4 * d) ||
        overlap(y, 4 * d, x_prev, 2 * d))
        return PROX_ERR_INVALID_ARG;
    return run_prox(layer, nullptr, keep_fraction, 0.5f, y, nullptr, nullptr, nullptr, nullptr,
                    reinterpret_cast<cudaStream_t>(stream), prox::kWaitLimitNs, 0, nullptr,
                    nullptr, x_prev, y_prev, x_out, eps);
}

prox_status prox_stack_ffn(const prox_layer* const* layers, int n_layers, const void* x0,
                           float keep_fraction, float eps, void* xs, float* ys,
                           prox_stream_t stream) {
    if (!layers || !x0 || !xs || !ys || n_layers < 1) return PROX_ERR_INVALID_ARG;
    if (n_layers > prox::kMaxStack) return PROX_ERR_UNSUPPORTED_SHAPE;
    if (!frac_ok(keep_fraction) || !(eps >= 0.0f) || !isfinite(eps)) return PROX_ERR_INVALID_ARG;
    const prox_layer* L0 = layers[0];
    if (!L0) return PROX_ERR_INVALID_ARG;
    if (!aligned16(x0) || !aligned16(xs) || !aligned16(ys)) return PROX_ERR_MISALIGNED;
    const size_t d = (size_t)L0->d_model, n = (size_t)n_layers;
    if (overlap(x0, 2 * d, xs, 2 * d * n) || overlap(x0, 2 * d, ys, 4 * d * n) ||
        overlap(xs, 2 * d * n, ys, 4 * d * n))
        return PROX_ERR_INVALID_ARG;
    prox::StackLayers sl;
    sl.n = n_layers;
    sl.x0 = static_cast<const uint16_t*>(x0);
    sl.xs = static_cast<uint16_t*>(xs);
    sl.ys = ys;
    for (int l = 0; l < n_layers; ++l) {
        const prox_layer* L = layers[l];
        if (!L) return PROX_ERR_INVALID_ARG;
        if (L->d_model != L0->d_model || L->d_ff != L0->d_ff || L->wq != L0->wq ||
            L->device != L0->device || L->num_blocks != L0->num_blocks)
            return PROX_ERR_INVALID_ARG;
        sl.layer[l].codes = L->codes;
        sl.layer[l].scales = L->scales;
        sl.layer[l].gateup = static_cast<const uint8_t*>(L->gateup);
        sl.layer[l].down_t = static_cast<const uint8_t*>(L->down_t);
    }
    prox::FusedLaunch f;
    f.codes = L0->codes;
    f.scales = L0->scales;
    f.gateup = L0->gateup;
    f.down_t = L0->down_t;
    f.wq = L0->wq;
    f.d = L0->d_model;
    f.F = L0->d_ff;
    f.x = sl.x0;
    f.y = ys;
    f.kx = prox_keep_count(L0->d_model, 0.5f);
    f.k = prox_keep_count(L0->d_ff, keep_fraction);
    f.eps = eps;
    f.ws = &L0->ws;  // the first layer's workspace serves the whole launch
    f.kept_out = nullptr;
    f.scores_out = nullptr;
    f.idx_out = nullptr;
    f.h_out = nullptr;
    f.num_blocks = L0->num_blocks;
    f.limit_ns = prox::kWaitLimitNs;
    f.inject = 0;
    f.ts = nullptr;
    return cuda_status(prox::launch_stack(f, sl, reinterpret_cast<cudaStream_t>(stream)));
}

prox_status prox_dense_ffn(const prox_layer* layer, const void* x, float* y,
                           prox_stream_t stream) {
    prox_status st = check_call(layer, x, y);
    if (st != PROX_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(y, 0, (size_t)layer->d_model * sizeof(float), s);
    if (e == cudaSuccess)
        e = prox::launch_dense(layer->gateup, layer->down_t, layer->wq,
                               static_cast<const uint16_t*>(x), layer->d_model, layer->d_ff, y,
                               layer->ws.status, layer->num_blocks, prox::kWaitLimitNs, nullptr,
                               s);
    return cuda_status(e);
}

prox_status prox_ffn_debug(const prox_layer* layer, const void* x, float keep_fraction,
                           float input_keep, float* y, int32_t* kept_inputs, float* scores,
                           int32_t* idx, float* h, prox_stream_t stream) {
    prox_status st = check_call(layer, x, y);
    if (st != PROX_OK) return st;
    if (!frac_ok(keep_fraction) || !frac_ok(input_keep)) return PROX_ERR_INVALID_ARG;
    const void* outs[] = {kept_inputs, scores, idx, h};
    for (const void* p : outs)
        if (p && !aligned16(p)) return PROX_ERR_MISALIGNED;
    return run_prox(layer, x, keep_fraction, input_keep, y, kept_inputs, scores, idx, h,
                    reinterpret_cast<cudaStream_t>(stream), prox::kWaitLimitNs, 0);
}

prox_status prox_ffn_batch(const prox_layer* layer, const void* x, int batch,
                           float keep_fraction, float* y, prox_stream_t stream) {
    prox_status st = check_call(layer, x, y);
    if (st != PROX_OK) return st;
    if (batch < 1 || !frac_ok(keep_fraction)) return PROX_ERR_INVALID_ARG;
    const size_t d = (size_t)layer->d_model;
    if ((d * 2) % 16 != 0) return PROX_ERR_MISALIGNED;  // every token's x 16-byte aligned
    const uint16_t* xs = static_cast<const uint16_t*>(x);
    // token t's own mask: one step per token, in order on the stream (the
    // layer's workspace is reused token after token)
    for (int t = 0; t < batch; ++t) {
        st = run_prox(layer, xs + (size_t)t * d, keep_fraction, 0.5f, y + (size_t)t * d, nullptr,
                      nullptr, nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream),
                      prox::kWaitLimitNs, 0);
        if (st != PROX_OK) return st;
    }
    return PROX_OK;
}

int prox_batch_union_group(const prox_layer* layer) {
    if (!layer || layer->wq) return 0;
    return prox::union_geometry(layer->d_model, layer->d_ff, layer->num_blocks).G;
}

namespace {

// A batch over the union of its tokens' masks, in passes of up to G tokens:
// clear the token bits, each token's mask-only step (its exact mask, its
// bit ORed into member[c]; y[t] zeroed), then Stage 2 over the union.
// member_out (debug, batch <= G): the token bits after the pass.
prox_status run_union(const prox_layer* L, const void* x, int batch, float keep_fraction,
                      float* y, uint32_t* member_out, cudaStream_t stream) {
    prox_status st = check_call(L, x, y);
    if (st != PROX_OK) return st;
    if (batch < 1 || !frac_ok(keep_fraction)) return PROX_ERR_INVALID_ARG;
    if (L->wq) return PROX_ERR_UNSUPPORTED_SHAPE;  // bf16 Stage-2 rows only
    const int G = prox_batch_union_group(L);
    if (G < 1) return PROX_ERR_UNSUPPORTED_SHAPE;
    if (member_out && (batch > G || !aligned16(member_out))) return PROX_ERR_INVALID_ARG;
    const size_t d = (size_t)L->d_model;
    if (overlap(x, 2 * d * batch, y, 4 * d * batch)) return PROX_ERR_INVALID_ARG;
    const uint16_t* xs = static_cast<const uint16_t*>(x);
    uint32_t* member = reinterpret_cast<uint32_t*>(L->ws.hch);  // debug h area, unused here
    // the proxy partials ([16][Fp] float2) are free after Stage 1: they hold
    // the union pass's partial g and u sums ([4][G][Fp] float, G <= 8)
    float* GU = reinterpret_cast<float*>(L->ws.part);
    const int k = prox_keep_count(L->d_ff, keep_fraction);
    const size_t part_bytes = (size_t)prox::kMaxSlices * prox::padded_ff(L->d_ff) * 8;
    // the grouped Stage-1 launch's barrier words, in the control block
    unsigned* gbar = reinterpret_cast<unsigned*>(reinterpret_cast<uint8_t*>(L->ws.status) + 1024);
    for (int g0 = 0; g0 < batch; g0 += G) {
        const int gb = std::min(G, batch - g0);
        cudaError_t e = cudaMemsetAsync(member, 0, (size_t)L->d_ff * 4, stream);
        if (e != cudaSuccess) return cuda_status(e);
        // Stage 1 of the pass's tokens: launches with a group of CTAs per
        // token, as many tokens per launch as the grid (a CTA per proxy tile
        // in every group) and the proxy-partial area (which the union pass
        // reuses afterwards) allow; a token left alone takes a mask-only step
        auto group_fits = [&](int nt) {
            const prox::MaskGroupGeom mg =
                prox::mask_group_geometry(L->d_model, L->d_ff, k, nt, L->num_blocks);
            return mg.gsize > 0 && (size_t)nt * mg.stride <= part_bytes;
        };
        for (int t = 0, nt = 0; t < gb; t += nt) {
            nt = gb - t;
            while (nt >= 2 && !group_fits(nt)) --nt;
            if (nt < 2) nt = 1;
            prox::FusedLaunch f;
            f.codes = L->codes;
            f.scales = L->scales;
            f.gateup = L->gateup;
            f.down_t = L->down_t;
            f.wq = 0;
            f.d = L->d_model;
            f.F = L->d_ff;
            f.x = xs + (g0 + t) * d;
            f.y = y + (g0 + t) * d;
            f.kx = prox_keep_count(L->d_model, 0.5f);
            f.k = k;
            f.member = member;
            f.token = t;
            f.ws = &L->ws;
            f.kept_out = nullptr;
            f.scores_out = nullptr;
            f.idx_out = nullptr;
            f.h_out = nullptr;
            f.num_blocks = L->num_blocks;
            f.limit_ns = prox::kWaitLimitNs;
            f.inject = 0;
            f.ts = nullptr;
            if (nt >= 2) {
                e = cudaMemsetAsync(gbar, 0, (size_t)nt * 4, stream);
                if (e == cudaSuccess)
                    e = prox::launch_masks(f, nt, t, reinterpret_cast<uint8_t*>(L->ws.part), gbar,
                                           stream);
            } else {
                e = prox::launch_fused(f, stream);
            }
            if (e != cudaSuccess) return cuda_status(e);
        }
        e = prox::launch_union(L->gateup, L->down_t, xs + g0 * d, member, GU, y + g0 * d,
                               L->d_model, L->d_ff, gb, L->num_blocks, L->ws.status,
                               prox::kWaitLimitNs, stream);
        if (e == cudaSuccess && member_out)
            e = cudaMemcpyAsync(member_out, member, (size_t)L->d_ff * 4, cudaMemcpyDeviceToDevice,
                                stream);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return PROX_OK;
}

}  // namespace

prox_status prox_ffn_batch_union(const prox_layer* layer, const void* x, int batch,
                                 float keep_fraction, float* y, prox_stream_t stream) {
    return run_union(layer, x, batch, keep_fraction, y, nullptr,
                     reinterpret_cast<cudaStream_t>(stream));
}

prox_status prox_ffn_batch_union_debug(const prox_layer* layer, const void* x, int batch,
                                       float keep_fraction, float* y, uint32_t* member_out,
                                       prox_stream_t stream) {
    if (!member_out) return PROX_ERR_INVALID_ARG;
    return run_union(layer, x, batch, keep_fraction, y, member_out,
                     reinterpret_cast<cudaStream_t>(stream));
}

prox_status prox_ffn_blocks(const prox_layer* layer, const void* x, int block_width,
                            float keep_fraction, float* y, prox_stream_t stream) {
    prox_status st = check_call(layer, x, y);
    if (st != PROX_OK) return st;
    if (!frac_ok(keep_fraction)) return PROX_ERR_INVALID_ARG;
    st = check_blocks(layer, block_width);
    if (st != PROX_OK) return st;
    return run_prox(layer, x, keep_fraction, 0.5f, y, nullptr, nullptr, nullptr, nullptr,
                    reinterpret_cast<cudaStream_t>(stream), prox::kWaitLimitNs, 0, nullptr,
                    nullptr, nullptr, nullptr, nullptr, 0.0f, block_width);
}

prox_status prox_ffn_blocks_debug(const prox_layer* layer, const void* x, int block_width,
                                  float keep_fraction, float* y, float* scores, int32_t* idx,
                                  float* h, prox_stream_t stream) {
    prox_status st = check_call(layer, x, y);
    if (st != PROX_OK) return st;
    if (!frac_ok(keep_fraction)) return PROX_ERR_INVALID_ARG;
    st = check_blocks(layer, block_width);
    if (st != PROX_OK) return st;
    const void* outs[] = {scores, idx, h};
    for (const void* p : outs)
        if (p && !aligned16(p)) return PROX_ERR_MISALIGNED;
    return run_prox(layer, x, keep_fraction, 0.5f, y, nullptr, scores, idx, h,
                    reinterpret_cast<cudaStream_t>(stream), prox::kWaitLimitNs, 0, nullptr,
                    nullptr, nullptr, nullptr, nullptr, 0.0f, block_width);
}

prox_status prox_ffn_contrib(const prox_layer* layer, const void* x, float keep_fraction, float* y,
                             prox_stream_t stream) {
    prox_status st = check_call(layer, x, y);
    if (st != PROX_OK) return st;
    if (!frac_ok(keep_fraction)) return PROX_ERR_INVALID_ARG;
    return run_prox(layer, x, keep_fraction, 0.5f, y, nullptr, nullptr, nullptr, nullptr,
                    reinterpret_cast<cudaStream_t>(stream), prox::kWaitLimitNs, 0, nullptr,
                    nullptr, nullptr, nullptr, nullptr, 0.0f, 0, true);
}

prox_status prox_ffn_contrib_debug(const prox_layer* layer, const void* x, float keep_fraction,
                                   float* y, float* scores, int32_t* idx, float* h,
                                   prox_stream_t stream) {
    prox_status st = check_call(layer, x, y);
    if (st != PROX_OK) return st;
    if (!frac_ok(keep_fraction)) return PROX_ERR_INVALID_ARG;
    const void* outs[] = {scores, idx, h};
    for (const void* p : outs)
        if (p && !aligned16(p)) return PROX_ERR_MISALIGNED;
    return run_prox(layer, x, keep_fraction, 0.5f, y, nullptr, scores, idx, h,
                    reinterpret_cast<cudaStream_t>(stream), prox::kWaitLimitNs, 0, nullptr,
                    nullptr, nullptr, nullptr, nullptr, 0.0f, 0, true);
}

prox_status prox_residual_rmsnorm(int d_model, const void* x, const float* y, float eps,
                                  void* x_next, prox_stream_t stream) {
    if (!x || !y || !x_next) return PROX_ERR_INVALID_ARG;
    if (d_model < 1 || d_model > prox::kMaxDModel) return PROX_ERR_UNSUPPORTED_SHAPE;
    if (!(eps >= 0.0f) || !isfinite(eps)) return PROX_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y) || !aligned16(x_next)) return PROX_ERR_MISALIGNED;
    return cuda_status(prox::launch_residual_rmsnorm(d_model, static_cast<const uint16_t*>(x), y,
                                                     eps, static_cast<uint16_t*>(x_next),
                                                     reinterpret_cast<cudaStream_t>(stream)));
}

prox_status prox_get_status(const prox_layer* layer, prox_stream_t stream) {
    if (!layer) return PROX_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, layer->ws.status, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    // clear the status word and, after a fault, the grid barrier word (a
    // barrier that ran out leaves it part-way)
    if (e == cudaSuccess)
        e = cudaMemsetAsync(layer->ws.status, 0, v != 0 ? prox::kControlBytes : sizeof(int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return PROX_ERR_CUDA;
    return (prox_status)v;
}

int prox_layer_blocks(const prox_layer* layer) { return layer ? layer->num_blocks : 0; }

prox_status prox_ffn_phase_times(const prox_layer* layer, const void* x, float keep_fraction,
                                 float* y, uint64_t* stamps, int dense, prox_stream_t stream) {
    prox_status st = check_call(layer, x, y);
    if (st != PROX_OK) return st;
    if (!stamps || (!dense && !frac_ok(keep_fraction))) return PROX_ERR_INVALID_ARG;
    if (!aligned16(stamps)) return PROX_ERR_MISALIGNED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(stamps, 0,
                                    (size_t)layer->num_blocks * PROX_PHASE_STAMPS * sizeof(uint64_t), s);
    if (e != cudaSuccess) return PROX_ERR_CUDA;
    if (dense) {
        e = cudaMemsetAsync(y, 0, (size_t)layer->d_model * sizeof(float), s);
        if (e == cudaSuccess)
            e = prox::launch_dense(layer->gateup, layer->down_t, layer->wq,
                                   static_cast<const uint16_t*>(x), layer->d_model, layer->d_ff,
                                   y, layer->ws.status, layer->num_blocks, prox::kWaitLimitNs,
                                   stamps, s);
        return cuda_status(e);
    }
    return run_prox(layer, x, keep_fraction, 0.5f, y, nullptr, nullptr, nullptr, nullptr, s,
                    prox::kWaitLimitNs, 0, nullptr, stamps);
}

prox_status prox_test_barrier_timeout(const prox_layer* layer, const void* x, float* y,
                                      prox_stream_t stream) {
    prox_status st = check_call(layer, x, y);
    if (st != PROX_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    st = run_prox(layer, x, 0.5f, 0.5f, y, nullptr, nullptr, nullptr, nullptr, s,
                  20 * 1000 * 1000LL /* 20 ms */, 1);
    if (st != PROX_OK) return st;
    return prox_get_status(layer, stream);
}

prox_status prox_layer_info(const prox_layer* layer, int* d_model, int* d_ff) {
    if (!layer) return PROX_ERR_INVALID_ARG;
    if (d_model) *d_model = layer->d_model;
    if (d_ff) *d_ff = layer->d_ff;
    return PROX_OK;
}

void prox_destroy(prox_layer* layer) { delete layer; }

}  // extern "C"
