/*
 * prox.h -- C ABI of libprox: two-stage sparse SwiGLU FFN decode (batch 1;
 * prox_ffn_batch runs a batch token by token) on NVIDIA B300 (sm_103a).
 * Variants of the same step: int8 or int4 Stage-2 rows (prox_prepare_q8,
 * prox_prepare_q4), block-
 * granular channel masks (prox_ffn_blocks), and the residual + RMSNorm glue
 * of a layer stack fused in front of the step (prox_ffn_resnorm).
 *
 * The method: "Prox: Training-Free FFN Activation Sparsity via Approximate
 * Intermediate-Channel Salience in LLMs", Abstract.  Stage 1 builds one
 * channel mask, shared by all three projections, from a sparsified input and
 * quantized proxy weights, keeping the channels whose approximate
 * intermediate-state magnitude ranks highest.  Stage 2 computes the selected
 * channels exactly.  The FFN itself is the SwiGLU block of "PrunePath:
 * Towards Highly Structured Sparse Language Models", Sec. 2.1 Eq. (1):
 *     FFN(x) = W_down ( silu(W_gate x) (.) (W_up x) )
 * (written there with x as a row vector; this library takes the nn.Linear
 * layouts below, i.e. the same product transposed).
 *
 * Readings the pages leave open, fixed here:
 *   - proxy: int4, symmetric, one fp16 scale per (channel, 128 input dims),
 *     s = fp16_rne(fl32(amax / 7)), q = clamp(rne(fl32(w / s)), -8, 7);
 *   - input sparsity: keep the ceil(input_keep * d) entries of largest |x|
 *     (ties -> lower index); default input_keep = 0.5;
 *   - ranking signal: score_c = |silu(g~_c) * u~_c| from the proxy state;
 *   - keep count: k = ceil(keep_fraction * d_ff) clamped to [1, d_ff]; the k
 *     highest scores win, ties -> lower channel;
 *   - Stage 2 uses the full (unsparsified) x; h and y are fp32.
 *
 * Conventions for every call:
 *   - Device memory is allocated and owned by the caller.  The library never
 *     allocates device memory and keeps no pointer to the source weights
 *     after prox_prepare returns.
 *   - Every call is ordered on the given CUDA stream (a cudaStream_t; NULL
 *     means the legacy default stream) and returns without synchronising,
 *     except prox_get_status.  prox_ffn needs no host read-back, so a
 *     sequence of calls can be captured in a CUDA graph.
 *   - Arguments are checked before any work is queued; a failed check
 *     returns an error code and queues nothing.  Launch failures return
 *     PROX_ERR_CUDA.  Faults found on the device (a bounded wait that ran
 *     out) are recorded in the layer's status word, read by
 *     prox_get_status.  No call traps, aborts or throws.
 *   - All device pointers must be 16-byte aligned.
 *   - Calls that share one prox_layer use its workspace and must be ordered
 *     with respect to each other (one stream, or events); calls on
 *     different layers are independent.
 *   - Shapes: d_model a multiple of 128 in [128, 10880] (the step's
 *     shared-memory tables must fit one SM); d_ff in [1, 32768]
 *     (prox_prepare also needs ceil(d_ff / #SMs) <= 256 and at most 256 SMs).
 *   - Inputs must be finite (no NaN or Inf in x or the weights).
 */
#ifndef PROX_H
#define PROX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of the ABI are exported even when the library is built with
 * hidden default visibility. */
#if defined(__GNUC__)
#define PROX_API __attribute__((visibility("default")))
#else
#define PROX_API
#endif

typedef struct CUstream_st* prox_stream_t; /* identical to cudaStream_t */

typedef enum prox_status {
    PROX_OK = 0,
    PROX_ERR_INVALID_ARG = 1,       /* null pointer, bad fraction, bad handle */
    PROX_ERR_UNSUPPORTED_SHAPE = 2, /* d_model / d_ff outside the limits above */
    PROX_ERR_MISALIGNED = 3,        /* a device pointer is not 16-byte aligned */
    PROX_ERR_CUDA = 4,              /* a CUDA runtime call or launch failed */
    PROX_ERR_TIMEOUT = 5,           /* a bounded on-device wait ran out */
    PROX_ERR_DEVICE_CHECK = 6       /* an on-device consistency check failed */
} prox_status;

/* Byte sizes of the caller-allocated device buffers for one layer. */
typedef struct prox_sizes {
    size_t proxy_codes;  /* int4 proxy codes, layout below */
    size_t proxy_scales; /* fp16 proxy scales, layout below */
    size_t gateup;       /* bf16 gate|up rows, [d_ff][2][d_model] */
    size_t down_t;       /* bf16 W_down transposed, [d_ff][d_model] */
    size_t workspace;    /* per-layer scratch used by prox_ffn */
} prox_sizes;

/* Opaque host-side handle: shapes plus the device pointers given to
 * prox_prepare.  Allocated by prox_prepare, released by prox_destroy. */
typedef struct prox_layer prox_layer;

/*
 * Device layouts written by prox_prepare (F = d_ff, d = d_model,
 * Fp = F rounded up to a multiple of 64, G = d / 128):
 *   proxy_codes  uint8 [d][Fp]: byte (j, c) = (q_gate[c][j] + 8)
 *                | (q_up[c][j] + 8) << 4, i.e. two offset-binary nibbles;
 *                input-dim-major so that one kept input j is one contiguous
 *                row; padding channels hold 0x88 (code 0).
 *   proxy_scales fp16  [G][Fp][2]: (s_gate[c][g], s_up[c][g]); padding 0.
 *   gateup       bf16  [F][2][d]: row c = (W_gate[c][:], W_up[c][:]).
 *   down_t       bf16  [F][d]:    row c = W_down[:][c].
 * prox_prepare_q8 writes int8 Stage-2 layouts instead of the last two.
 * Every Stage-2 row r (W_gate[c], W_up[c], W_down[:][c]) is quantized
 * symmetrically on its own: s_r = fl32(max_j |r_j| / 127) and
 * q_r[j] = clamp(rne(fl32(r_j / s_r)), -127, 127), q_r = 0 where s_r = 0:
 *   gateup_q8    [F] rows of 2 d + 16 bytes: int8 q_gate[c][0..d),
 *                int8 q_up[c][0..d), then fp32 s_gate[c], s_up[c],
 *                s_down[c] and 4 zero bytes.
 *   down_q8      int8 [F][d]: row c = q_down[c][:], the codes of W_down[:][c].
 * prox_prepare_q4 writes int4 Stage-2 layouts the same way with
 * s_r = fl32(max_j |r_j| / 7) and q_r[j] = clamp(rne(fl32(r_j / s_r)), -8, 7),
 * packed as offset-binary nibbles n = q + 8, eight consecutive elements
 * 8 i .. 8 i + 7 per little-endian 32-bit word i, element 8 i + 2 m + h in
 * bits 16 h + 4 m (m = 0..3, h = 0..1):
 *   gateup_q4    [F] rows of d + 16 bytes: d / 8 words of q_gate[c],
 *                d / 8 words of q_up[c], then fp32 s_gate[c], s_up[c],
 *                s_down[c] and 4 zero bytes.
 *   down_q4      [F] rows of d / 2 bytes: the words of q_down[c][:].
 */

/* Sizes of the buffers above for a layer shape.  Host only; queues nothing.
 * Returns PROX_ERR_UNSUPPORTED_SHAPE for shapes outside the limits. */
PROX_API prox_status prox_query_sizes(int d_model, int d_ff, prox_sizes* out);

/* As prox_query_sizes for prox_prepare_q8: gateup and down_t hold the sizes
 * of gateup_q8 (d_ff * (2 d_model + 16)) and down_q8 (d_ff * d_model). */
PROX_API prox_status prox_query_sizes_q8(int d_model, int d_ff, prox_sizes* out);

/* As prox_query_sizes for prox_prepare_q4: gateup and down_t hold the sizes
 * of gateup_q4 (d_ff * (d_model + 16)) and down_q4 (d_ff * d_model / 2). */
PROX_API prox_status prox_query_sizes_q4(int d_model, int d_ff, prox_sizes* out);

/*
 * One-off per-layer preparation ("Prox", Abstract: quantized proxy weights
 * for Stage 1; Stage-2 layouts for the selected rows and columns).
 *   w_gate, w_up : bf16 [d_ff][d_model] (nn.Linear weight layout), device
 *   w_down       : bf16 [d_model][d_ff], device
 *   proxy_codes, proxy_scales, gateup, down_t, workspace : device buffers of
 *                  at least the sizes prox_query_sizes reports; written here
 *                  (workspace is zeroed) and referenced by the handle.
 * On success *out receives a new handle.  The source weights may be freed
 * once the stream has passed this call.  Not timed; not for graph capture
 * (it sets kernel attributes).
 */
PROX_API prox_status prox_prepare(int d_model, int d_ff, const void* w_gate, const void* w_up,
                         const void* w_down, void* proxy_codes, void* proxy_scales,
                         void* gateup, void* down_t, void* workspace, prox_stream_t stream,
                         prox_layer** out);

/*
 * As prox_prepare, with int8 Stage-2 weights ("Prox", Abstract: the method
 * composes with weight quantization; here the selected rows themselves are
 * int8, which halves the Stage-2 bytes per channel): gateup_q8
 * and down_q8 (sizes from prox_query_sizes_q8) receive the int8 layouts
 * above; the proxy is the same.  Every step entry point (prox_ffn, _ex,
 * _host, _traced, _resnorm, _debug, _noalloc, _batch, _blocks,
 * prox_dense_ffn, prox_ffn_phase_times) then runs Stage 2 on the int8 rows:
 *   g_c = s_gate[c] sum_j q_gate[c][j] x_j,  u_c likewise,
 *   y   = sum_{c in mask} silu(g_c) u_c s_down[c] q_down[c][:]
 * in fp32 (each code-times-bf16 product is exact).  The channel mask is the
 * one of the bf16 layer: it depends on the proxy only.
 */
PROX_API prox_status prox_prepare_q8(int d_model, int d_ff, const void* w_gate, const void* w_up,
                            const void* w_down, void* proxy_codes, void* proxy_scales,
                            void* gateup_q8, void* down_q8, void* workspace,
                            prox_stream_t stream, prox_layer** out);

/*
 * As prox_prepare_q8 with int4 Stage-2 rows (a quarter of the bf16 bytes per
 * channel): gateup_q4 and down_q4 (sizes from prox_query_sizes_q4) receive
 * the int4 layouts above.  The same entry points run on the layer, with the
 * same sums over the int4 codes; the channel mask is again the bf16 layer's.
 * Errors as prox_prepare.
 */
PROX_API prox_status prox_prepare_q4(int d_model, int d_ff, const void* w_gate, const void* w_up,
                            const void* w_down, void* proxy_codes, void* proxy_scales,
                            void* gateup_q4, void* down_q4, void* workspace,
                            prox_stream_t stream, prox_layer** out);

/*
 * The Prox decode step ("Prox", Abstract; Eq. (1) of the PrunePath page for
 * Stage 2), input keep fixed at 0.5:
 *   x             bf16 [d_model], device
 *   keep_fraction FFN keep fraction rho in (0, 1]; k = ceil(rho * d_ff)
 *   y             fp32 [d_model], device, overwritten with
 *                 y = sum_{c in mask} W_down[:, c] * silu(W_gate[c] . x) * (W_up[c] . x)
 */
PROX_API prox_status prox_ffn(const prox_layer* layer, const void* x, float keep_fraction, float* y,
                     prox_stream_t stream);

/* As prox_ffn with an explicit input keep fraction in (0, 1]:
 * k_x = ceil(input_keep * d_model) inputs feed the proxy. */
PROX_API prox_status prox_ffn_ex(const prox_layer* layer, const void* x, float keep_fraction,
                        float input_keep, float* y, prox_stream_t stream);

/*
 * prox_ffn with host buffers, for callers whose token lives in host memory:
 * copies x_host (bf16 [d_model]) to a staging slot of the layer's
 * workspace, runs the decode step there (input keep 0.5) and copies y (fp32
 * [d_model]) back to y_host.  All three steps are queued on the stream; the
 * call does not synchronise, so y_host is valid once the stream has passed
 * the call.  Pass page-locked host memory (cudaHostAlloc / pinned tensors)
 * for asynchronous copies; pageable memory still works but the runtime then
 * copies synchronously.  No alignment rule applies to the host pointers.
 */
PROX_API prox_status prox_ffn_host(const prox_layer* layer, const void* x_host, float keep_fraction,
                          float* y_host, prox_stream_t stream);

/* Number of CUDA events prox_ffn_traced records. */
#define PROX_TRACE_EVENTS 2

/*
 * prox_ffn_ex that also records `events` (n_events == PROX_TRACE_EVENTS
 * cudaEvent_t handles, created by the caller with timing enabled) around its
 * kernel: the decode step is one persistent kernel, so
 * cudaEventElapsedTime(events[0], events[1]) is its duration on the stream.
 * Inside a stream capture the records become event nodes of the graph
 * (cudaEventRecordExternal).  For timing only; it launches the same kernel
 * as prox_ffn_ex.
 */
PROX_API prox_status prox_ffn_traced(const prox_layer* layer, const void* x, float keep_fraction,
                            float input_keep, float* y, void* const* events, int n_events,
                            prox_stream_t stream);

/* Number of phase timestamps per CTA written by prox_ffn_phase_times. */
#define PROX_PHASE_STAMPS 16

/* Number of CTAs (one per SM) the layer's kernels launch.  Host only. */
PROX_API int prox_layer_blocks(const prox_layer* layer);

/*
 * Tracing: one decode step (dense == 0, input keep 0.5) or one dense step
 * (dense != 0, keep_fraction ignored) that also stores, per CTA b, the
 * device clock (%globaltimer, ns) at its phase boundaries into
 * stamps[b * PROX_PHASE_STAMPS + i] (uint64, device, prox_layer_blocks()
 * rows, zeroed first; a phase the kernel does not have stays 0):
 *   0 start; 1 input selection done; 2 proxy partials written;
 *   3 past the first grid barrier; 4 scores, histogram counts and score
 *   keys published; 5 exact channel mask known (this CTA's item list
 *   final, Stage 2 starts); 6 first gate|up row landed; 7 gate|up dot
 *   products done; 8 W_down^T accumulation done; 9 end; 10 input-magnitude
 *   histogram built; 11 first proxy row landed (thread 0); 12 proxy loop
 *   done (thread 0); 13 scores formed; 14 past the second grid barrier,
 *   first 11-bit digit of the k-th score key known; 15 exact k-th score
 *   key found (digits 2 and 3).
 * The dense step stamps 0 and 6..9 only.  Same results as prox_ffn /
 * prox_dense_ffn.
 */
PROX_API prox_status prox_ffn_phase_times(const prox_layer* layer, const void* x,
                                 float keep_fraction, float* y, uint64_t* stamps, int dense,
                                 prox_stream_t stream);

/*
 * Batch > 1 decode with per-token masks: for each of the `batch` tokens
 * x[t] (bf16 [batch][d_model], rows contiguous, device) its own Prox step
 * (Stage 1 mask of that token, Stage 2 on its selected channels) writes
 * y[t] (fp32 [batch][d_model], device); keep fraction as in prox_ffn.  The
 * steps run one after another on the stream (one persistent launch per
 * token).  Identical to prox_ffn called per token.
 */
PROX_API prox_status prox_ffn_batch(const prox_layer* layer, const void* x, int batch,
                           float keep_fraction, float* y, prox_stream_t stream);

/*
 * Batch > 1 decode over the union of the tokens' masks.  Every token keeps
 * its own exact mask and output, as in prox_ffn_batch ("Prox", Abstract: one
 * channel mask per token from its proxy ranking; y[t] = the SwiGLU block of
 * "PrunePath", Sec. 2.1 Eq. (1), over token t's selected channels only), but
 * Stage 2 reads each row in the union of the masks once for all the tokens
 * whose mask holds it.  The batch runs in passes of prox_batch_union_group()
 * tokens: a mask-only step per token (Stage 1, its bit ORed into a
 * per-channel word), then one gate|up pass and one W_down^T pass over the
 * union.  Where the tokens' Stage-1 scratch fits in the layer's workspace
 * (the Llama shapes), the pass's mask-only steps run as one launch with a
 * group of CTAs per token.  x bf16 [batch][d_model], y fp32 [batch][d_model] (device, 16-byte
 * aligned, not overlapping); keep fraction as in prox_ffn.  The same masks
 * as prox_ffn per token; y[t] equals prox_ffn's up to the order of the fp32
 * additions.  Layers prepared with int8 or int4 Stage-2 rows
 * (prox_prepare_q8, _q4) are not supported (PROX_ERR_UNSUPPORTED_SHAPE).  Uses the layer's workspace.
 */
PROX_API prox_status prox_ffn_batch_union(const prox_layer* layer, const void* x, int batch,
                                 float keep_fraction, float* y, prox_stream_t stream);

/* Tokens per pass of prox_ffn_batch_union on this layer (their x fit in a
 * CTA's shared memory next to the gate|up ring): 8 up to d_model 4096,
 * fewer above; 0 for a null, int8 or int4 layer. */
PROX_API int prox_batch_union_group(const prox_layer* layer);

/* prox_ffn_batch_union plus, for batch <= prox_batch_union_group(),
 * member_out (uint32 [d_ff], device): bit t of word c is set when token t's
 * mask holds channel c (parity checks). */
PROX_API prox_status prox_ffn_batch_union_debug(const prox_layer* layer, const void* x,
                                       int batch, float keep_fraction, float* y,
                                       uint32_t* member_out, prox_stream_t stream);

/*
 * The decode step with a block-granular mask ("PrunePath", Sec. 2.2 Eq. (2):
 * after a channel permutation, d_ff splits into E = d_ff / block_width
 * contiguous experts; Sec. 3.1 runs a subset of them).  The weights given to
 * prox_prepare are taken as already permuted.  Stage 1 is unchanged; the
 * score of expert e is the sum of its channels' proxy scores (fp32, fixed
 * order); the K = ceil(keep_fraction E) experts of largest score are kept
 * (ties -> lower expert) and Stage 2 runs over all their channels
 * (k = K block_width), so its rows are read in contiguous runs.
 *   block_width  a power of two in [4, 256] (else PROX_ERR_INVALID_ARG)
 *                dividing d_ff, with E >= the layer's CTA count and every
 *                CTA's share of whole blocks <= 256 channels (else
 *                PROX_ERR_UNSUPPORTED_SHAPE): e.g. 4..64 for d_ff 14336 on
 *                148 SMs.
 * x, y and the input keep (0.5) as in prox_ffn.
 */
PROX_API prox_status prox_ffn_blocks(const prox_layer* layer, const void* x, int block_width,
                            float keep_fraction, float* y, prox_stream_t stream);

/* prox_ffn_blocks plus, for parity checks, the per-channel proxy scores
 * (fp32 [d_ff], before the block sums), the selected channels (int32 [k],
 * ascending) and h (fp32 [k], idx order); each may be NULL. */
PROX_API prox_status prox_ffn_blocks_debug(const prox_layer* layer, const void* x,
                                  int block_width, float keep_fraction, float* y,
                                  float* scores, int32_t* idx, float* h,
                                  prox_stream_t stream);

/*
 * The decode step with a second selection signal, after the COUNTDOWN page
 * ("COUNTDOWN", Abstract): the FFN output is a linear combination of the
 * down projection's columns, y = sum_c h_c W_down[:, c], and its
 * predictor-free variant ranks channels by indirect coefficients.  Here
 * channel c is ranked by the magnitude of its term of that combination,
 *   score_c = |silu(g~_c) u~_c| * ||W_down[:, c]||_2,
 * with g~, u~ the Prox proxy state (Stage 1 as in prox_ffn) and the column
 * norms computed in fp32 by prox_prepare (kept in the layer's workspace);
 * the k = ceil(rho d_ff) largest are kept (ties to the lower channel) and
 * Stage 2 is prox_ffn's.  x bf16 [d_model], y fp32 [d_model], both device;
 * input keep 0.5.  Same status and ordering rules as prox_ffn.
 */
PROX_API prox_status prox_ffn_contrib(const prox_layer* layer, const void* x, float keep_fraction,
                                      float* y, prox_stream_t stream);

/* prox_ffn_contrib plus the contribution scores (fp32 [d_ff]), the channel
 * list (int32 [k], ascending) and h (fp32 [k], in list order); any of the
 * three may be NULL; non-NULL ones 16-byte aligned (parity checks). */
PROX_API prox_status prox_ffn_contrib_debug(const prox_layer* layer, const void* x,
                                            float keep_fraction, float* y, float* scores,
                                            int32_t* idx, float* h, prox_stream_t stream);

/*
 * A stack of n_layers decode steps in ONE persistent launch (the stacked
 * residual-stream workload: x_{l+1} = RMSNorm(x_l + y_l), no learned gain):
 *   layer 0 runs prox_ffn on x0; layer l > 0 runs it on
 *   x_l = bf16_rne((x_{l-1} + y_{l-1}) / sqrt(mean((x_{l-1} + y_{l-1})^2) + eps)),
 *   computed inside layer l's own step; a grid barrier between layers makes
 *   y_{l-1} complete before layer l reads it, so no launch separates them.
 *   layers   host array of n_layers handles of one shape (d_model, d_ff, the
 *            same Stage-2 format and device); 1 <= n_layers <= 64
 *            (PROX_ERR_UNSUPPORTED_SHAPE beyond); the launch uses
 *            layers[0]'s workspace and status word (prox_get_status(layers[0]))
 *   x0       bf16 [d_model], device: layer 0's input
 *   xs       bf16 [n_layers][d_model], device: row l receives x_l (l >= 1;
 *            row 0 is left as it is)
 *   ys       fp32 [n_layers][d_model], device: row l receives y_l
 * keep_fraction in (0, 1] for every layer, input keep 0.5, eps >= 0.  x0, xs
 * and ys must not overlap (PROX_ERR_INVALID_ARG); all 16-byte aligned.
 * The layers' workspaces other than the first are not touched; calls that
 * share layers[0] must be ordered as for prox_ffn.
 */
PROX_API prox_status prox_stack_ffn(const prox_layer* const* layers, int n_layers, const void* x0,
                                    float keep_fraction, float eps, void* xs, float* ys,
                                    prox_stream_t stream);

/* Dense SwiGLU FFN, Eq. (1) of the PrunePath page over all d_ff channels,
 * streaming the same gateup / down_t buffers (the in-library dense
 * baseline).  x bf16 [d_model], y fp32 [d_model], both device. */
PROX_API prox_status prox_dense_ffn(const prox_layer* layer, const void* x, float* y,
                           prox_stream_t stream);

/*
 * prox_ffn_ex plus the intermediate results, for parity checks (not timed).
 * Each extra output may be NULL; all are device buffers:
 *   kept_inputs int32 [k_x]  kept input indices, ascending
 *   scores      fp32  [d_ff] proxy ranking signal |silu(g~) u~| per channel
 *   idx         int32 [k]    selected channels, ascending
 *   h           fp32  [k]    Stage-2 intermediate state h_c, in idx order
 */
PROX_API prox_status prox_ffn_debug(const prox_layer* layer, const void* x, float keep_fraction,
                           float input_keep, float* y, int32_t* kept_inputs, float* scores,
                           int32_t* idx, float* h, prox_stream_t stream);

/*
 * Glue between stacked layers (no page defines it; plain reading of a
 * residual stream): z = x + y, x_next = bf16_rne(z / sqrt(mean(z^2) + eps)),
 * no learned gain.  x, x_next bf16 [d_model]; y fp32 [d_model]; device.
 * x_next may not alias y.
 */
PROX_API prox_status prox_residual_rmsnorm(int d_model, const void* x, const float* y, float eps,
                                  void* x_next, prox_stream_t stream);

/*
 * One layer of a stack with the glue fused into the step (the pages define
 * no glue; plain reading of a residual stream, as prox_residual_rmsnorm):
 * x = bf16_rne(z / sqrt(mean(z^2) + eps)) with z = x_prev + y_prev, then
 * y = prox_ffn(layer, x, keep_fraction).  Every CTA of the step computes x
 * itself (in the same order, so all agree); x is also written to x_out for
 * the next layer's residual.  Saves the separate glue launch per layer.
 *   x_prev bf16 [d_model], y_prev fp32 [d_model] (the previous layer's input
 *   and output), x_out bf16 [d_model], y fp32 [d_model]; all device, 16-byte
 *   aligned.  x_out and y must not overlap x_prev, y_prev or each other
 *   (PROX_ERR_INVALID_ARG).  Same status and ordering rules as prox_ffn.
 */
PROX_API prox_status prox_ffn_resnorm(const prox_layer* layer, const void* x_prev,
                                      const float* y_prev, float eps, void* x_out,
                                      float keep_fraction, float* y, prox_stream_t stream);

/*
 * prox_ffn without any caller-provided scratch (the pages have no
 * counterpart: this is a deployment variant).  For callers that cannot
 * allocate device memory when they run a step -- a host framework or server
 * that reserved the device up front and refuses further allocations, plugins
 * and latency-critical loops where an allocation would synchronise the
 * device -- the step's scratch (proxy partials, score histogram, score
 * keys, grid-barrier words) lives in a fixed 4 MiB array compiled into the
 * library, which every device that loads the library holds until the process
 * exits.  Nothing is allocated: no cudaMalloc, cudaFree or allocating
 * library routine is called.
 *   x  bf16 [d_model], device; keep_fraction in (0, 1] (input keep 0.5);
 *   y  fp32 [d_model], device, overwritten as by prox_ffn.
 * Limits and rules:
 *   - the layer's workspace (prox_query_sizes().workspace) must fit in
 *     4 MiB: every d_ff up to 28544 at any supported d_model does, so the
 *     Llama-2-7B and Llama-3-8B shapes do; d_ff 28672 fits up to d_model
 *     9216, so the Llama-3-70B shape (d_model 8192) does too; larger layers
 *     return PROX_ERR_UNSUPPORTED_SHAPE and queue nothing;
 *   - the layer's device must be the current device (else
 *     PROX_ERR_INVALID_ARG);
 *   - the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture;
 *   - every call on a device shares the array and finds the previous call's
 *     contents (the call clears what must start at zero); calls that overlap
 *     on the GPU race and must be ordered by the caller;
 *   - device-side faults are recorded in the layer's status word, as for
 *     prox_ffn (prox_get_status).
 */
PROX_API prox_status prox_ffn_noalloc(const prox_layer* layer, const void* x, float keep_fraction,
                             float* y, prox_stream_t stream);

/* Synchronises the stream, returns the status recorded on the device by
 * earlier calls on this layer (PROX_OK if none) and clears it.  After a
 * fault it also resets the layer's grid-barrier word, so later calls on the
 * layer run normally again. */
PROX_API prox_status prox_get_status(const prox_layer* layer, prox_stream_t stream);

/*
 * Failure-detection test hook (not for production use): runs one decode
 * step in which one CTA withholds its arrival at the grid barrier and
 * every bounded wait gives up after 20 ms, then synchronises and returns
 * the layer's status, which is PROX_ERR_TIMEOUT when the bounded waits work
 * (the status and barrier words are reset as by prox_get_status).  y is
 * left undefined.  x bf16 [d_model], y fp32 [d_model], both device.
 */
PROX_API prox_status prox_test_barrier_timeout(const prox_layer* layer, const void* x, float* y,
                                      prox_stream_t stream);

/* Shapes of a prepared layer.  Host only. */
PROX_API prox_status prox_layer_info(const prox_layer* layer, int* d_model, int* d_ff);

/* k = ceil(frac * n) in fp64, clamped to [1, n]; 0 for n < 1 or a fraction
 * outside (0, 1].  Host only. */
PROX_API int prox_keep_count(int n, float frac);

/* Releases the host handle only; the device buffers stay the caller's. */
PROX_API void prox_destroy(prox_layer* layer);

/* Static description of a status code. */
PROX_API const char* prox_status_string(prox_status status);

#ifdef __cplusplus
}
#endif

#endif /* PROX_H */
