/*
 * prox_oracle.c -- plain, slow CPU oracle for the Prox sparse SwiGLU FFN
 * decode step.  TEST INFRASTRUCTURE ONLY: it is compiled and called by the
 * tests, by the package's smoke check and by the CPU-baseline leg of the
 * benchmark, never by the product path.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * Sources followed (cited by page title and section):
 *   [Prox]  "Prox: Training-Free FFN Activation Sparsity via Approximate
 *           Intermediate-Channel Salience in LLMs", Abstract: Stage 1 builds
 *           one shared channel mask from a sparsified input and quantized
 *           proxy weights, ranking channels by the magnitude of the
 *           approximate intermediate state; Stage 2 computes the selected
 *           channels exactly, so all three projections run sparse.
 *   [PP]    "PrunePath: Towards Highly Structured Sparse Language Models",
 *           Sec. 2.1 Eq. (1): FFN(x) = (phi(x W_gate) (.) x W_up) W_down,
 *           phi = SiLU, h = phi(x W_gate) (.) x W_up element-wise along d_ff.
 *
 * Every number the pages leave open is a stated reading (the int4 group-128
 * symmetric proxy, the top-|x| input keep, the |silu(g~) u~| score, ceil for
 * the keep count, lowest-index tie-breaks, fp16 scale storage).  Each
 * function names its reading.
 *
 * Arithmetic: fp64 everywhere, except the quantizer, whose scale and code
 * rounding are defined in fp32 by the reading (so that the codes are a
 * well-defined integer result).  Weights and activations come in as raw
 * bf16 bit patterns (uint16), in nn.Linear layouts:
 *   W_gate, W_up : [F][d]   (row c = intermediate channel c)
 *   W_down       : [d][F]   (row i = output element i)
 * which is Eq. (1) transposed (the page writes x as a row vector).
 *
 * Pins: every function here is checked by the CPU tests against something
 * other than itself (numpy's float16 rounding, exhaustive sorting, closed
 * forms, invariants and special cases).  Nothing here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1

/* ------------------------------------------------------------------------ */
/* Number formats                                                           */
/* ------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32 pattern. */
double oracle_bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* binary16 value from its fields: sign, 5-bit exponent (bias 15), 10-bit
 * fraction; exponent 0 = subnormal (fraction * 2^-24), 31 = inf/nan. */
double oracle_fp16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp(1.0 + (double)m / 1024.0, e - 15);
    }
    return sign ? -v : v;
}

/* Round a binary32 value to the nearest binary16 value, ties to even, and
 * return it as a double.  In the binade [2^E, 2^(E+1)) binary16 values are
 * multiples of 2^(E-10); below 2^-14 (subnormals) the spacing stays 2^-24.
 * Results above the largest finite value 65504 become infinity. */
double oracle_round_to_fp16(float f) {
    double v = (double)f;
    if (isnan(v)) return v;
    double a = fabs(v);
    if (isinf(a)) return v;
    if (a == 0.0) return v;
    int e2;
    frexp(a, &e2);          /* a = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;         /* a in [2^E, 2^(E+1)) */
    if (E < -14) E = -14;
    double quantum = ldexp(1.0, E - 10);
    double n = nearbyint(a / quantum);  /* exact quotient; default mode is RNE */
    double r = n * quantum;
    if (r > 65504.0) r = INFINITY;
    return v < 0 ? -r : r;
}

/* Round a double to the nearest bf16 (8 significant bits), ties to even,
 * returning the bf16 bit pattern.  Used only for the residual/RMSNorm glue
 * between stacked layers. */
uint16_t oracle_double_to_bf16(double v) {
    if (isnan(v)) return 0x7fc0;
    double a = fabs(v);
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);
    int E = e2 - 1;
    if (E < -126) E = -126;
    double quantum = ldexp(1.0, E - 7);
    double r = nearbyint(a / quantum) * quantum;
    /* largest finite bf16 = (2 - 2^-7) * 2^127 */
    if (r > ldexp(2.0 - ldexp(1.0, -7), 127)) return sign | 0x7f80;
    float f = (float)r; /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7fff));
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

double oracle_silu(double z) { return silu(z); }

/* Keep count for a fraction: ceil(frac * n) computed in fp64 on the fraction
 * as given (a binary32), clamped to [1, n].  Reading: the pages give no rule;
 * ceil keeps at least the requested fraction. */
int oracle_keep_count(int n, float frac) {
    double k = ceil((double)frac * (double)n);
    if (k < 1.0) k = 1.0;
    if (k > (double)n) k = (double)n;
    return (int)k;
}

/* ------------------------------------------------------------------------ */
/* a0: quantized proxy weights ([Prox] Abstract, "quantized proxy weights") */
/* ------------------------------------------------------------------------ */
/* Reading: int4, symmetric, one scale per (output channel, group of 128
 * consecutive input dims).  For channel c, group g:
 *   amax = max |W[c][j]| over the group (binary32, exact)
 *   s    = fp16_rne(fl32(amax / 7))
 *   q_j  = clamp(rne(fl32(W[c][j] / s)), -8, 7), or 0 when s == 0.
 * Outputs: q[F][d] int8 codes, s[F][G] scales as doubles (each an fp16
 * value, G = d / 128). */
int oracle_quantize(int F, int d, const uint16_t* W, int8_t* q, double* s) {
    if (F <= 0 || d <= 0 || d % 128 != 0 || !W || !q || !s) return ORACLE_BAD_ARG;
    int G = d / 128;
    for (int c = 0; c < F; ++c) {
        for (int g = 0; g < G; ++g) {
            float amax = 0.0f;
            for (int t = 0; t < 128; ++t) {
                float w = (float)oracle_bf16_to_double(W[(size_t)c * d + g * 128 + t]);
                float aw = fabsf(w);
                if (aw > amax) amax = aw;
            }
            float s32 = amax / 7.0f;                 /* binary32 division */
            double sv = oracle_round_to_fp16(s32);
            s[(size_t)c * G + g] = sv;
            float sf = (float)sv;                    /* exact */
            for (int t = 0; t < 128; ++t) {
                size_t at = (size_t)c * d + g * 128 + t;
                int code = 0;
                if (sf != 0.0f) {
                    float w = (float)oracle_bf16_to_double(W[at]);
                    float ratio = w / sf;            /* binary32 division */
                    float r = rintf(ratio);          /* ties to even */
                    if (r < -8.0f) r = -8.0f;
                    if (r > 7.0f) r = 7.0f;
                    code = (int)r;
                }
                q[at] = (int8_t)code;
            }
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Top-k selection by magnitude with the lowest index winning ties.         */
/* ------------------------------------------------------------------------ */
typedef struct { double key; int index; } ranked;

static int by_key_desc_index_asc(const void* pa, const void* pb) {
    const ranked* a = (const ranked*)pa;
    const ranked* b = (const ranked*)pb;
    if (a->key > b->key) return -1;
    if (a->key < b->key) return 1;
    return (a->index > b->index) - (a->index < b->index);
}

static int by_index(const void* pa, const void* pb) {
    int a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    return (a > b) - (a < b);
}

/* Sort (key desc, index asc), keep the first k, return them in ascending
 * index order.  The library sort is the only step. */
static int topk_ascending(int n, const double* key, int k, int32_t* out) {
    if (n <= 0 || k < 0 || k > n) return ORACLE_BAD_ARG;
    ranked* r = (ranked*)malloc(sizeof(ranked) * (size_t)n);
    if (!r) return ORACLE_BAD_ARG;
    for (int i = 0; i < n; ++i) { r[i].key = key[i]; r[i].index = i; }
    qsort(r, (size_t)n, sizeof(ranked), by_key_desc_index_asc);
    for (int i = 0; i < k; ++i) out[i] = r[i].index;
    qsort(out, (size_t)k, sizeof(int32_t), by_index);
    free(r);
    return ORACLE_OK;
}

/* a1: input sparsity ([Prox] Abstract, "uses input sparsity").  Reading:
 * keep the kx entries of x with the largest |x_j| (ties -> lower j; -0 and
 * +0 are equal); the sparsified input x~ is x on the kept set, 0 elsewhere.
 * Output: kept indices, ascending. */
int oracle_input_topk(int d, const uint16_t* x, int kx, int32_t* kept) {
    if (d <= 0 || !x || !kept || kx < 1 || kx > d) return ORACLE_BAD_ARG;
    double* mag = (double*)malloc(sizeof(double) * (size_t)d);
    if (!mag) return ORACLE_BAD_ARG;
    for (int j = 0; j < d; ++j) mag[j] = fabs(oracle_bf16_to_double(x[j]));
    int rc = topk_ascending(d, mag, kx, kept);
    free(mag);
    return rc;
}

/* a2: proxy intermediate state and ranking signal ([Prox] Abstract: Stage 1
 * approximates the SwiGLU intermediate state from x~ and the quantized proxy
 * weights; only the magnitude ranking of its entries is used).
 *   g~_c = sum_{j in kept} s_gate[c][j/128] * q_gate[c][j] * x_j
 *   u~_c = sum_{j in kept} s_up[c][j/128]   * q_up[c][j]   * x_j
 *   score_c = | silu(g~_c) * u~_c |
 * all in fp64.  Any of ghat/uhat may be NULL. */
int oracle_proxy_scores(int F, int d,
                        const int8_t* q_gate, const double* s_gate,
                        const int8_t* q_up, const double* s_up,
                        const uint16_t* x, int kx, const int32_t* kept,
                        double* ghat, double* uhat, double* score) {
    if (F <= 0 || d <= 0 || d % 128 != 0 || kx < 1 || kx > d || !q_gate || !s_gate ||
        !q_up || !s_up || !x || !kept || !score)
        return ORACLE_BAD_ARG;
    int G = d / 128;
    for (int c = 0; c < F; ++c) {
        double g = 0.0, u = 0.0;
        for (int t = 0; t < kx; ++t) {
            int j = kept[t];
            double xj = oracle_bf16_to_double(x[j]);
            size_t at = (size_t)c * d + j;
            g += s_gate[(size_t)c * G + j / 128] * (double)q_gate[at] * xj;
            u += s_up[(size_t)c * G + j / 128] * (double)q_up[at] * xj;
        }
        if (ghat) ghat[c] = g;
        if (uhat) uhat[c] = u;
        score[c] = fabs(silu(g) * u);
    }
    return ORACLE_OK;
}

/* a3: the shared channel mask ([Prox] Abstract: mask from the magnitude
 * ranking).  Reading: the k channels with the largest score (ties -> lower
 * channel), emitted in ascending channel order. */
/* Second selection signal, COUNTDOWN style ("COUNTDOWN", Abstract: the
 * FFN output is a linear combination of the down projection's columns,
 * y = sum_c h_c W_down[:, c], whose coefficients carry the sparsity;
 * M-COUNTDOWN ranks by indirect, predictor-free coefficients).  Reading: the
 * proxy's approximate coefficient magnitude |h~_c| = state_score[c] weighted
 * by the norm of the column it scales, i.e. the magnitude of that term of
 * the linear combination:  out[c] = state_score[c] * ||W_down[:, c]||_2,
 * with the norm in fp64 over the bf16 column.  (D-COUNTDOWN's trained
 * predictor of the direct coefficients is out of scope.) */
int oracle_contrib_scores(int F, int d, const uint16_t* w_down, const double* state_score,
                          double* out) {
    if (F <= 0 || d <= 0 || !w_down || !state_score || !out) return ORACLE_BAD_ARG;
    for (int c = 0; c < F; ++c) {
        double ss = 0.0;
        for (int i = 0; i < d; ++i) {
            double w = oracle_bf16_to_double(w_down[(size_t)i * F + c]);
            ss += w * w;
        }
        out[c] = state_score[c] * sqrt(ss);
    }
    return ORACLE_OK;
}

int oracle_channel_topk(int F, const double* score, int k, int32_t* idx) {
    if (!score || !idx) return ORACLE_BAD_ARG;
    return topk_ascending(F, score, k, idx);
}

/* f3: block-granular mask ([PP] Sec. 2.2 Eq. (2): after a permutation the
 * intermediate dimension splits into E = F / bw contiguous experts of width
 * bw, and the FFN is the sum of the experts' outputs; Sec. 3.1 activates a
 * subset of experts).  Reading for the training-free Prox signal: the score
 * of expert e is the sum of its channels' scores,
 *   S_e = sum_{c = e bw}^{(e+1) bw - 1} score_c   (fp64, channel order),
 * the K experts with the largest S_e are kept (ties -> lower expert), and
 * the mask is every channel of those experts, in ascending channel order
 * (K bw channels).  The permutation is the identity: the weights passed in
 * are taken to be already permuted.  block_score (length E) may be NULL. */
int oracle_block_topk(int F, const double* score, int bw, int K, double* block_score,
                      int32_t* idx) {
    if (F <= 0 || !score || !idx || bw < 1 || F % bw != 0) return ORACLE_BAD_ARG;
    int E = F / bw;
    if (K < 1 || K > E) return ORACLE_BAD_ARG;
    double* S = (double*)malloc(sizeof(double) * (size_t)E);
    int32_t* blocks = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
    if (!S || !blocks) {
        free(S);
        free(blocks);
        return ORACLE_BAD_ARG;
    }
    for (int e = 0; e < E; ++e) {
        double acc = 0.0;
        for (int t = 0; t < bw; ++t) acc += score[(size_t)e * bw + t];
        S[e] = acc;
        if (block_score) block_score[e] = acc;
    }
    int rc = topk_ascending(E, S, K, blocks);
    if (rc == ORACLE_OK)
        for (int i = 0; i < K; ++i)
            for (int t = 0; t < bw; ++t) idx[(size_t)i * bw + t] = blocks[i] * bw + t;
    free(S);
    free(blocks);
    return rc;
}

/* a4-a5: Stage 2 ([Prox] Abstract: selected channels computed exactly;
 * [PP] Eq. (1)).  For c in idx (any order, no repeats):
 *   g_c = W_gate[c] . x,  u_c = W_up[c] . x,  h_c = silu(g_c) * u_c
 *   y_i = sum_{c in idx} W_down[i][c] * h_c
 * with the full bf16 x (reading: "exactly" means the unsparsified input).
 * h (length k, in idx order) may be NULL. */
int oracle_sparse_ffn(int F, int d, const uint16_t* w_gate, const uint16_t* w_up,
                      const uint16_t* w_down, const uint16_t* x, int k,
                      const int32_t* idx, double* h, double* y) {
    if (F <= 0 || d <= 0 || k < 0 || k > F || !w_gate || !w_up || !w_down || !x || !y ||
        (k > 0 && !idx))
        return ORACLE_BAD_ARG;
    for (int i = 0; i < d; ++i) y[i] = 0.0;
    for (int t = 0; t < k; ++t) {
        int c = idx[t];
        if (c < 0 || c >= F) return ORACLE_BAD_ARG;
        double g = 0.0, u = 0.0;
        for (int j = 0; j < d; ++j) {
            double xj = oracle_bf16_to_double(x[j]);
            g += oracle_bf16_to_double(w_gate[(size_t)c * d + j]) * xj;
            u += oracle_bf16_to_double(w_up[(size_t)c * d + j]) * xj;
        }
        double hc = silu(g) * u;
        if (h) h[t] = hc;
        for (int i = 0; i < d; ++i) y[i] += oracle_bf16_to_double(w_down[(size_t)i * F + c]) * hc;
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Next row (int8 Stage-2 weights): [Prox] Abstract, the method is          */
/* "compatible with quantization"; the scheme is a reading.                 */
/* ------------------------------------------------------------------------ */
/* Symmetric int8, one fp32 scale per row of a [rows][n] bf16 matrix:
 *   amax = max_j |W[r][j]| (binary32, exact), s = fl32(amax / 127),
 *   q_j  = clamp(rne(fl32(W[r][j] / s)), -127, 127), or 0 when s == 0.
 * Stage 2 quantizes the rows of W_gate and W_up and the rows of W_down^T
 * (the columns of W_down). */
int oracle_quantize_rows_q8(int rows, int n, const uint16_t* W, int8_t* q, float* s) {
    if (rows <= 0 || n <= 0 || !W || !q || !s) return ORACLE_BAD_ARG;
    for (int r = 0; r < rows; ++r) {
        float amax = 0.0f;
        for (int j = 0; j < n; ++j) {
            float aw = fabsf((float)oracle_bf16_to_double(W[(size_t)r * n + j]));
            if (aw > amax) amax = aw;
        }
        float sr = amax / 127.0f;                    /* binary32 division */
        s[r] = sr;
        for (int j = 0; j < n; ++j) {
            int code = 0;
            if (sr != 0.0f) {
                float w = (float)oracle_bf16_to_double(W[(size_t)r * n + j]);
                float t = rintf(w / sr);             /* binary32 division, ties to even */
                if (t < -127.0f) t = -127.0f;
                if (t > 127.0f) t = 127.0f;
                code = (int)t;
            }
            q[(size_t)r * n + j] = (int8_t)code;
        }
    }
    return ORACLE_OK;
}

/* Symmetric int4, one fp32 scale per row (the int4 reading of the same
 * sentence): amax as above, s = fl32(amax / 7),
 *   q_j = clamp(rne(fl32(W[r][j] / s)), -8, 7), or 0 when s == 0
 * (|w / s| <= 7, so -8 is never reached from a symmetric scale; the clamp
 * is the int4 range).  The codes are returned as int8 values in [-8, 7]. */
int oracle_quantize_rows_q4(int rows, int n, const uint16_t* W, int8_t* q, float* s) {
    if (rows <= 0 || n <= 0 || !W || !q || !s) return ORACLE_BAD_ARG;
    for (int r = 0; r < rows; ++r) {
        float amax = 0.0f;
        for (int j = 0; j < n; ++j) {
            float aw = fabsf((float)oracle_bf16_to_double(W[(size_t)r * n + j]));
            if (aw > amax) amax = aw;
        }
        float sr = amax / 7.0f;                      /* binary32 division */
        s[r] = sr;
        for (int j = 0; j < n; ++j) {
            int code = 0;
            if (sr != 0.0f) {
                float w = (float)oracle_bf16_to_double(W[(size_t)r * n + j]);
                float t = rintf(w / sr);             /* binary32 division, ties to even */
                if (t < -8.0f) t = -8.0f;
                if (t > 7.0f) t = 7.0f;
                code = (int)t;
            }
            q[(size_t)r * n + j] = (int8_t)code;
        }
    }
    return ORACLE_OK;
}

/* Stage 2 on int8 weights ([PP] Eq. (1) with the dequantized rows): for c in
 * idx, g_c = s_gate[c] sum_j q_gate[c][j] x_j, u_c likewise,
 * h_c = silu(g_c) u_c, y_i = sum_c h_c s_down[c] q_down[c][i], where
 * q_down / s_down quantize the rows of W_down^T.  fp64, full bf16 x.  The
 * same sums serve int4 codes (values in [-8, 7] held as int8). */
int oracle_sparse_ffn_q8(int F, int d, const int8_t* q_gate, const float* s_gate,
                         const int8_t* q_up, const float* s_up, const int8_t* q_down,
                         const float* s_down, const uint16_t* x, int k, const int32_t* idx,
                         double* h, double* y) {
    if (F <= 0 || d <= 0 || k < 0 || k > F || !q_gate || !s_gate || !q_up || !s_up ||
        !q_down || !s_down || !x || !y || (k > 0 && !idx))
        return ORACLE_BAD_ARG;
    for (int i = 0; i < d; ++i) y[i] = 0.0;
    for (int t = 0; t < k; ++t) {
        int c = idx[t];
        if (c < 0 || c >= F) return ORACLE_BAD_ARG;
        double g = 0.0, u = 0.0;
        for (int j = 0; j < d; ++j) {
            double xj = oracle_bf16_to_double(x[j]);
            g += (double)q_gate[(size_t)c * d + j] * xj;
            u += (double)q_up[(size_t)c * d + j] * xj;
        }
        g *= (double)s_gate[c];
        u *= (double)s_up[c];
        double hc = silu(g) * u;
        if (h) h[t] = hc;
        double hs = hc * (double)s_down[c];
        for (int i = 0; i < d; ++i) y[i] += hs * (double)q_down[(size_t)c * d + i];
    }
    return ORACLE_OK;
}

/* a6: the dense SwiGLU FFN, [PP] Eq. (1), written directly: the intermediate
 * state h over all channels, then the down projection row by row. */
int oracle_dense_ffn(int F, int d, const uint16_t* w_gate, const uint16_t* w_up,
                     const uint16_t* w_down, const uint16_t* x, double* h, double* y) {
    if (F <= 0 || d <= 0 || !w_gate || !w_up || !w_down || !x || !y) return ORACLE_BAD_ARG;
    double* hh = (double*)malloc(sizeof(double) * (size_t)F);
    if (!hh) return ORACLE_BAD_ARG;
    for (int c = 0; c < F; ++c) {
        double g = 0.0, u = 0.0;
        for (int j = 0; j < d; ++j) {
            double xj = oracle_bf16_to_double(x[j]);
            g += oracle_bf16_to_double(w_gate[(size_t)c * d + j]) * xj;
            u += oracle_bf16_to_double(w_up[(size_t)c * d + j]) * xj;
        }
        hh[c] = silu(g) * u;
        if (h) h[c] = hh[c];
    }
    for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int c = 0; c < F; ++c) acc += oracle_bf16_to_double(w_down[(size_t)i * F + c]) * hh[c];
        y[i] = acc;
    }
    free(hh);
    return ORACLE_OK;
}

/* The whole two-stage step ([Prox] Abstract), in the pages' order: input
 * sparsity, proxy state from the quantized weights, the shared mask from its
 * magnitude ranking, then exact Stage 2 on the mask.  Outputs other than y
 * may be NULL. */
int oracle_prox_ffn(int F, int d, const uint16_t* w_gate, const uint16_t* w_up,
                    const uint16_t* w_down, const int8_t* q_gate, const double* s_gate,
                    const int8_t* q_up, const double* s_up, const uint16_t* x, int kx, int k,
                    int32_t* kept_out, double* score_out, int32_t* idx_out, double* h_out,
                    double* y) {
    if (F <= 0 || d <= 0 || kx < 1 || kx > d || k < 1 || k > F || !y) return ORACLE_BAD_ARG;
    int32_t* kept = (int32_t*)malloc(sizeof(int32_t) * (size_t)kx);
    double* score = (double*)malloc(sizeof(double) * (size_t)F);
    int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
    int rc = ORACLE_BAD_ARG;
    if (!kept || !score || !idx) goto done;
    rc = oracle_input_topk(d, x, kx, kept);
    if (rc) goto done;
    rc = oracle_proxy_scores(F, d, q_gate, s_gate, q_up, s_up, x, kx, kept, NULL, NULL, score);
    if (rc) goto done;
    rc = oracle_channel_topk(F, score, k, idx);
    if (rc) goto done;
    rc = oracle_sparse_ffn(F, d, w_gate, w_up, w_down, x, k, idx, h_out, y);
    if (rc) goto done;
    if (kept_out) memcpy(kept_out, kept, sizeof(int32_t) * (size_t)kx);
    if (score_out) memcpy(score_out, score, sizeof(double) * (size_t)F);
    if (idx_out) memcpy(idx_out, idx, sizeof(int32_t) * (size_t)k);
done:
    free(kept);
    free(score);
    free(idx);
    return rc;
}

/* Glue between stacked layers (no page defines it; reading): the residual
 * z = x + y, then RMS normalisation without a learned gain,
 *   x_next = bf16_rne( z / sqrt(mean(z^2) + eps) ). */
int oracle_residual_rmsnorm(int d, const uint16_t* x, const double* y, double eps,
                            uint16_t* x_next) {
    if (d <= 0 || !x || !y || !x_next) return ORACLE_BAD_ARG;
    double ss = 0.0;
    double* z = (double*)malloc(sizeof(double) * (size_t)d);
    if (!z) return ORACLE_BAD_ARG;
    for (int i = 0; i < d; ++i) {
        z[i] = oracle_bf16_to_double(x[i]) + y[i];
        ss += z[i] * z[i];
    }
    double inv = 1.0 / sqrt(ss / (double)d + eps);
    for (int i = 0; i < d; ++i) x_next[i] = oracle_double_to_bf16(z[i] * inv);
    free(z);
    return ORACLE_OK;
}
