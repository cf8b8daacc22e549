/*
 * CPU oracle for the routed-expert RVQ MoE step.  TEST INFRASTRUCTURE ONLY:
 * only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg may load it.  It shares no code, header or table with the CUDA
 * library, and the library never calls it.
 *
 * Plain, slow, single-threaded C.  Inputs are the fp32 / uint8 arrays the
 * method stores; every sum is carried in double.  Each function states the
 * passage it follows.  Sources (web pages about the WASTE engine):
 *   [fr]  "Exécuter Kimi K3 avec 29 Go de RAM à 0,50 tok/s"
 *   [vi]  "Chạy Kimi K3 ở 0.50 tok/s với 29GB RAM"  (same text, Vietnamese)
 * Where the pages leave a step open, the reading taken is stated at the
 * function.
 *
 * Logical code layout used throughout (one matrix with n_out rows and
 * n_in = 8*nv inputs): codes[r][s][j], r < n_out, s < 3 stages, j < nv,
 * i.e. byte (r*3 + s)*nv + j.  Vector j of row r covers inputs 8j..8j+7.
 * Codebooks of one matrix: cb[s][c][v], s < 3, c < 256, v < 8, fp32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_STAGES 3
#define OR_K 256
#define OR_V 8

static size_t code_index(int nv, int r, int s, int j) {
    return ((size_t)r * OR_STAGES + (size_t)s) * (size_t)nv + (size_t)j;
}

static double cb_at(const float *cb, int s, int c, int v) {
    return (double)cb[((size_t)s * OR_K + (size_t)c) * OR_V + (size_t)v];
}

/*
 * Dequantise one matrix ([fr] "Quantification et exactitude": residual
 * vector quantisation in 3 stages, 256-entry codebooks of 8-dimensional
 * vectors).  Reading: the stages are residuals, so a weight vector is the
 * sum of the three selected codebook vectors; the sum is taken in double
 * (exact for three fp32 addends of these magnitudes up to rounding at 2^-53).
 * W is row-major [n_out][n_in].
 */
void oracle_dequant(int n_out, int n_in, const float *cb, const uint8_t *codes, double *W) {
    int nv = n_in / OR_V;
    for (int r = 0; r < n_out; ++r)
        for (int j = 0; j < nv; ++j)
            for (int v = 0; v < OR_V; ++v) {
                double w = 0.0;
                for (int s = 0; s < OR_STAGES; ++s)
                    w += cb_at(cb, s, codes[code_index(nv, r, s, j)], v);
                W[(size_t)r * n_in + (size_t)j * OR_V + v] = w;
            }
}

/* y = W x, plain row-by-row dot products in double. */
void oracle_matvec_dense(int n_out, int n_in, const double *W, const double *x, double *y) {
    for (int r = 0; r < n_out; ++r) {
        double acc = 0.0;
        for (int i = 0; i < n_in; ++i) acc += W[(size_t)r * n_in + i] * x[i];
        y[r] = acc;
    }
}

/*
 * The pages' product without rebuilding the matrix ([fr] "Quantification et
 * exactitude": a table of partial dot products is built, then every row
 * costs 3 table lookups and 2 additions per vector).  Table entry
 * T[s][j][c] = <cb[s][c][:], x[8j..8j+7]>; row r accumulates
 * T[0][j][c0] + T[1][j][c1] + T[2][j][c2] over its vectors j.
 */
void oracle_matvec_lut(int n_out, int n_in, const float *cb, const uint8_t *codes,
                       const double *x, double *y) {
    int nv = n_in / OR_V;
    double *T = (double *)malloc(sizeof(double) * (size_t)OR_STAGES * (size_t)nv * OR_K);
    if (!T) return;
    for (int s = 0; s < OR_STAGES; ++s)
        for (int j = 0; j < nv; ++j)
            for (int c = 0; c < OR_K; ++c) {
                double t = 0.0;
                for (int v = 0; v < OR_V; ++v) t += cb_at(cb, s, c, v) * x[(size_t)j * OR_V + v];
                T[((size_t)s * nv + j) * OR_K + c] = t;
            }
    for (int r = 0; r < n_out; ++r) {
        double acc = 0.0;
        for (int j = 0; j < nv; ++j) {
            double t0 = T[((size_t)0 * nv + j) * OR_K + codes[code_index(nv, r, 0, j)]];
            double t1 = T[((size_t)1 * nv + j) * OR_K + codes[code_index(nv, r, 1, j)]];
            double t2 = T[((size_t)2 * nv + j) * OR_K + codes[code_index(nv, r, 2, j)]];
            acc += t0 + t1 + t2;
        }
        y[r] = acc;
    }
    free(T);
}

/*
 * Router logits l[e] = sum_i W_r[e][i] h[i] + b[e] ([fr] "Lecture anticipée
 * et prédiction du routeur": the router of a layer decides the expert IDs).
 * bias may be NULL (no bias).
 */
void oracle_router(int n_experts, int d, const float *Wr, const float *bias, const double *h,
                   double *logits) {
    for (int e = 0; e < n_experts; ++e) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += (double)Wr[(size_t)e * d + i] * h[i];
        logits[e] = acc + (bias ? (double)bias[e] : 0.0);
    }
}

/* true when expert a ranks before expert b: larger logit first, lower index on ties */
static int ranks_before(const double *l, int a, int b) {
    if (l[a] > l[b]) return 1;
    if (l[a] < l[b]) return 0;
    return a < b;
}

/*
 * Top-k selection and gate normalisation.  The pages give 16 expert IDs per
 * token and layer ([fr] "Lecture anticipée ..."); the order (logit
 * descending, lowest index first on equal logits) and the softmax over the
 * k selected logits are the readings taken where the pages are silent.
 * Selection is a plain k-pass scan; idx comes out in rank order.
 */
void oracle_topk_softmax(int n_experts, int k, const double *logits, int32_t *idx, double *gate) {
    unsigned char *taken = (unsigned char *)calloc((size_t)n_experts, 1);
    if (!taken) return;
    for (int i = 0; i < k; ++i) {
        int best = -1;
        for (int e = 0; e < n_experts; ++e) {
            if (taken[e]) continue;
            if (best < 0 || ranks_before(logits, e, best)) best = e;
        }
        taken[best] = 1;
        idx[i] = best;
    }
    double lmax = logits[idx[0]];
    double z = 0.0;
    for (int i = 0; i < k; ++i) z += exp(logits[idx[i]] - lmax);
    for (int i = 0; i < k; ++i) gate[i] = exp(logits[idx[i]] - lmax) / z;
    free(taken);
}

/* silu(z) = z / (1 + e^-z) */
double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * One expert's FFN on one token: a = silu(G x) * (U x), y = D a.  The three
 * matrices gate, up and down are the ones the pages store side by side in
 * one record ([fr] "Architecture de streaming depuis le disque"); SwiGLU is
 * the reading taken for how they combine.  cb holds the expert's codebooks
 * [3 matrices: gate, up, down][3][256][8]; use_lut selects the table form
 * (1) or dequantise-then-multiply (0).
 */
void oracle_expert_ffn(int d, int f, const float *cb, const uint8_t *gate_codes,
                       const uint8_t *up_codes, const uint8_t *down_codes, const double *x,
                       double *y, int use_lut) {
    const size_t cb_mat = (size_t)OR_STAGES * OR_K * OR_V;
    double *zg = (double *)malloc(sizeof(double) * (size_t)f);
    double *zu = (double *)malloc(sizeof(double) * (size_t)f);
    double *a = (double *)malloc(sizeof(double) * (size_t)f);
    if (!zg || !zu || !a) { free(zg); free(zu); free(a); return; }
    if (use_lut) {
        oracle_matvec_lut(f, d, cb + 0 * cb_mat, gate_codes, x, zg);
        oracle_matvec_lut(f, d, cb + 1 * cb_mat, up_codes, x, zu);
    } else {
        double *W = (double *)malloc(sizeof(double) * (size_t)f * (size_t)d);
        if (!W) { free(zg); free(zu); free(a); return; }
        oracle_dequant(f, d, cb + 0 * cb_mat, gate_codes, W);
        oracle_matvec_dense(f, d, W, x, zg);
        oracle_dequant(f, d, cb + 1 * cb_mat, up_codes, W);
        oracle_matvec_dense(f, d, W, x, zu);
        free(W);
    }
    for (int r = 0; r < f; ++r) a[r] = oracle_silu(zg[r]) * zu[r];
    if (use_lut) {
        oracle_matvec_lut(d, f, cb + 2 * cb_mat, down_codes, a, y);
    } else {
        double *W = (double *)malloc(sizeof(double) * (size_t)d * (size_t)f);
        if (!W) { free(zg); free(zu); free(a); return; }
        oracle_dequant(d, f, cb + 2 * cb_mat, down_codes, W);
        oracle_matvec_dense(d, f, W, a, y);
        free(W);
    }
    free(zg); free(zu); free(a);
}

/*
 * Gate-weighted combine of the k expert outputs of one token:
 * out[i] = base[i] + sum_k gate[k] * ys[k][i], k in rank order.  base may be
 * NULL (zero).  The residual form h + combine is the reading taken for how a
 * layer's output feeds the next layer.
 */
void oracle_combine(int d, int k, const double *gate, const double *ys, const double *base,
                    double *out) {
    for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int t = 0; t < k; ++t) acc += gate[t] * ys[(size_t)t * d + i];
        out[i] = (base ? base[i] : 0.0) + acc;
    }
}

/*
 * One MoE layer over T tokens with every expert's arrays in memory:
 * per token, router -> top-k + softmax -> k expert FFNs -> combine.
 * h [T][d] (double), cbs [E][3][3][256][8], codes in the logical layout per
 * expert: gate/up [E][f][3][d/8], down [E][d][3][f/8].  residual != 0 adds
 * h to the output.  logits [T][E], idx [T][k], gate [T][k] are outputs.
 */
void oracle_moe_layer(int T, int d, int f, int n_experts, int k, const float *Wr,
                      const float *bias, const float *cbs, const uint8_t *gate_codes,
                      const uint8_t *up_codes, const uint8_t *down_codes, const double *h,
                      int residual, int use_lut, double *out, double *logits, int32_t *idx,
                      double *gate) {
    const size_t cb_exp = (size_t)3 * OR_STAGES * OR_K * OR_V;
    const size_t gu_exp = (size_t)f * OR_STAGES * (size_t)(d / OR_V);
    const size_t dn_exp = (size_t)d * OR_STAGES * (size_t)(f / OR_V);
    double *ys = (double *)malloc(sizeof(double) * (size_t)k * (size_t)d);
    if (!ys) return;
    for (int t = 0; t < T; ++t) {
        const double *ht = h + (size_t)t * d;
        double *lt = logits + (size_t)t * n_experts;
        oracle_router(n_experts, d, Wr, bias, ht, lt);
        oracle_topk_softmax(n_experts, k, lt, idx + (size_t)t * k, gate + (size_t)t * k);
        for (int i = 0; i < k; ++i) {
            int e = idx[(size_t)t * k + i];
            oracle_expert_ffn(d, f, cbs + (size_t)e * cb_exp, gate_codes + (size_t)e * gu_exp,
                              up_codes + (size_t)e * gu_exp, down_codes + (size_t)e * dn_exp, ht,
                              ys + (size_t)i * d, use_lut);
        }
        oracle_combine(d, k, gate + (size_t)t * k, ys, residual ? ht : NULL,
                       out + (size_t)t * d);
    }
    free(ys);
}

/*
 * Weightless RMS normalisation out = in / sqrt(mean(in^2) + 1e-6).  Not one of
 * the pages' operations: it stands in for the trunk's normalisation of each
 * MoE layer's input when layers are chained as h <- h + MoE(norm(h)) (the
 * plain chain h <- h + MoE(h) diverges at the test workloads' scales).
 */
void oracle_rmsnorm(int d, const double *in, double *out) {
    double ss = 0.0;
    for (int i = 0; i < d; ++i) ss += in[i] * in[i];
    double scale = 1.0 / sqrt(ss / (double)d + 1e-6);
    for (int i = 0; i < d; ++i) out[i] = in[i] * scale;
}

/*
 * One layer of the decode chain, applied in place to h [T][d]: per token,
 * x = rmsnorm(h_t) feeds the router and the experts, and the gate-weighted
 * combine is added back, h_t <- h_t + sum_i g_i y_i(x).  The pages stack 92
 * MoE layers per token, each layer's routing decided on the hidden state the
 * previous layer left ([fr] "Budget RAM et zone de performance étroite": 16
 * experts x 92 layers per token; "Lecture anticipée et prédiction du
 * routeur": layer L+1's router reads layer L's residual).  The residual add
 * is the pages' "h += combine"; the norm in front of the layer stands in for
 * the trunk, which is out of scope (see oracle_rmsnorm).  Arrays as in
 * oracle_moe_layer; logits [T][E], idx [T][k], gate [T][k] are outputs.
 */
void oracle_residual_layer(int T, int d, int f, int n_experts, int k, const float *Wr,
                           const float *bias, const float *cbs, const uint8_t *gate_codes,
                           const uint8_t *up_codes, const uint8_t *down_codes, double *h,
                           int use_lut, double *logits, int32_t *idx, double *gate) {
    const size_t cb_exp = (size_t)3 * OR_STAGES * OR_K * OR_V;
    const size_t gu_exp = (size_t)f * OR_STAGES * (size_t)(d / OR_V);
    const size_t dn_exp = (size_t)d * OR_STAGES * (size_t)(f / OR_V);
    double *x = (double *)malloc(sizeof(double) * (size_t)d);
    double *ys = (double *)malloc(sizeof(double) * (size_t)k * (size_t)d);
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    if (!x || !ys || !y) { free(x); free(ys); free(y); return; }
    for (int t = 0; t < T; ++t) {
        double *ht = h + (size_t)t * d;
        double *lt = logits + (size_t)t * n_experts;
        int32_t *it = idx + (size_t)t * k;
        double *gt = gate + (size_t)t * k;
        oracle_rmsnorm(d, ht, x);
        oracle_router(n_experts, d, Wr, bias, x, lt);
        oracle_topk_softmax(n_experts, k, lt, it, gt);
        for (int i = 0; i < k; ++i) {
            int e = it[i];
            oracle_expert_ffn(d, f, cbs + (size_t)e * cb_exp, gate_codes + (size_t)e * gu_exp,
                              up_codes + (size_t)e * gu_exp, down_codes + (size_t)e * dn_exp, x,
                              ys + (size_t)i * d, use_lut);
        }
        oracle_combine(d, k, gt, ys, NULL, y);
        for (int i = 0; i < d; ++i) ht[i] = ht[i] + y[i];
    }
    free(x); free(ys); free(y);
}

/*
 * Bytes of codes per expert: 3 matrices (gate, up, down) of d*f weights at
 * 3 stages x 1 byte per 8 weights = 3.00 bits per weight ([fr]
 * "Quantification et exactitude").
 */
uint64_t oracle_expert_code_bytes(int d, int f) {
    return (uint64_t)3 * (uint64_t)OR_STAGES * (uint64_t)d * (uint64_t)f / OR_V;
}

/*
 * crc32 of a byte string as the record check uses it ([fr] "Architecture de streaming
 * depuis le disque": crc32 behind --verify): IEEE 802.3 / zlib -- reflected polynomial
 * 0xEDB88320, register preset to all ones, result complemented -- one bit at a time.
 */
uint32_t oracle_crc32(const uint8_t *p, size_t n) {
    uint32_t c = 0xFFFFFFFFu;
    for (size_t i = 0; i < n; ++i) {
        c ^= p[i];
        for (int b = 0; b < 8; ++b) c = (c >> 1) ^ (0xEDB88320u & (0u - (c & 1u)));
    }
    return ~c;
}

/*
 * RVQ encoder: codes and codebooks for a dense matrix ([fr] "Quantification et exactitude":
 * 3 residual stages of 256 eight-dimensional vectors; the pages' converter is named there but
 * its training is not described).  Reading taken -- greedy residual k-means:
 *   the residual R starts as W; for stage s = 0, 1, 2:
 *     C[c] = R[init[s][c]] for c < 256 (vector indices drawn by the caller);
 *     `iters` Lloyd rounds: every vector goes to its nearest centroid, then every centroid
 *       with members becomes their mean (an empty one keeps its value);
 *     one more assignment with the final C gives the stage's codes, and R <- R - C[code].
 * Nearest: least d(x, c) = sum over v = 0..7 of (x_v - c_v)^2, accumulated in that order in
 *   fp32 with one fused multiply-add per term (a code is an integer decided by floating point,
 *   so the device takes it in the same precision); ties go to the lower index.
 * Mean: each member component in fixed point, q = round-to-nearest(x * 2^40) as int64, so
 *   the sums are exact in any order; mean = (float)(((double)sum / count) * 2^-40).
 * Vector j of row r of W [rows][cols] (fp32 row-major) covers columns 8j..8j+7; it is vector
 * r*nv + j.  cb [3][256][8]; codes [rows][3][nv]; err[s] = sum of the squared residual
 * components after stage s (double, in vector order).  Returns 0, or -1 when cols % 8 != 0,
 * an init index is out of range, or a weight is not finite or has |w| >= 2^22.
 */
#define OR_FIX 1099511627776.0 /* 2^40 */

int oracle_rvq_nearest(const float *x, const float *C) {
    int best = 0;
    float bd = INFINITY;
    for (int c = 0; c < OR_K; ++c) {
        float d = 0.0f;
        for (int v = 0; v < OR_V; ++v) {
            float t = x[v] - C[(size_t)c * OR_V + v];
            d = fmaf(t, t, d);
        }
        if (d < bd) {
            bd = d;
            best = c;
        }
    }
    return best;
}

static void rvq_means(size_t n, const float *R, const uint8_t *code, float *C) {
    int64_t sum[OR_K][OR_V];
    int64_t cnt[OR_K];
    memset(sum, 0, sizeof sum);
    memset(cnt, 0, sizeof cnt);
    for (size_t i = 0; i < n; ++i) {
        int c = code[i];
        cnt[c] += 1;
        for (int v = 0; v < OR_V; ++v) sum[c][v] += (int64_t)llrint((double)R[i * OR_V + v] * OR_FIX);
    }
    for (int c = 0; c < OR_K; ++c) {
        if (cnt[c] == 0) continue;
        for (int v = 0; v < OR_V; ++v)
            C[(size_t)c * OR_V + v] = (float)(((double)sum[c][v] / (double)cnt[c]) * (1.0 / OR_FIX));
    }
}

/* codes of one stage with the stage's codebook C, then R <- R - C[code]; returns sum R^2 */
static double rvq_apply_stage(size_t n, float *R, const float *C, uint8_t *code) {
    double e = 0.0;
    for (size_t i = 0; i < n; ++i) {
        int c = oracle_rvq_nearest(R + i * OR_V, C);
        code[i] = (uint8_t)c;
        for (int v = 0; v < OR_V; ++v) {
            R[i * OR_V + v] = R[i * OR_V + v] - C[(size_t)c * OR_V + v];
            e += (double)R[i * OR_V + v] * (double)R[i * OR_V + v];
        }
    }
    return e;
}

static int rvq_check(int rows, int cols, const float *W) {
    if (rows < 0 || cols < 0 || cols % OR_V) return -1;
    for (size_t i = 0; i < (size_t)rows * (size_t)cols; ++i)
        if (!(fabsf(W[i]) < 4194304.0f)) return -1; /* also refuses NaN */
    return 0;
}

static void rvq_scatter_codes(int rows, int nv, int s, const uint8_t *code, uint8_t *codes) {
    for (int r = 0; r < rows; ++r)
        for (int j = 0; j < nv; ++j) codes[code_index(nv, r, s, j)] = code[(size_t)r * nv + j];
}

int oracle_rvq_train(int rows, int cols, const float *W, const int32_t *init, int iters, float *cb,
                     uint8_t *codes, double *err) {
    if (rvq_check(rows, cols, W) || iters < 0) return -1;
    const int nv = cols / OR_V;
    const size_t n = (size_t)rows * (size_t)nv;
    for (int i = 0; i < OR_STAGES * OR_K; ++i)
        if (init[i] < 0 || (size_t)init[i] >= n) return -1;
    float *R = malloc(n * OR_V * sizeof(float) + 1);
    uint8_t *code = malloc(n + 1);
    if (!R || !code) {
        free(R);
        free(code);
        return -1;
    }
    memcpy(R, W, n * OR_V * sizeof(float));
    for (int s = 0; s < OR_STAGES; ++s) {
        float *C = cb + (size_t)s * OR_K * OR_V;
        for (int c = 0; c < OR_K; ++c)
            for (int v = 0; v < OR_V; ++v) C[(size_t)c * OR_V + v] = R[(size_t)init[s * OR_K + c] * OR_V + v];
        for (int it = 0; it < iters; ++it) {
            for (size_t i = 0; i < n; ++i) code[i] = (uint8_t)oracle_rvq_nearest(R + i * OR_V, C);
            rvq_means(n, R, code, C);
        }
        err[s] = rvq_apply_stage(n, R, C, code);
        rvq_scatter_codes(rows, nv, s, code, codes);
    }
    free(R);
    free(code);
    return 0;
}

/* The three final assignments alone, with given codebooks cb [3][256][8]. */
int oracle_rvq_encode(int rows, int cols, const float *W, const float *cb, uint8_t *codes, double *err) {
    if (rvq_check(rows, cols, W)) return -1;
    const int nv = cols / OR_V;
    const size_t n = (size_t)rows * (size_t)nv;
    float *R = malloc(n * OR_V * sizeof(float) + 1);
    uint8_t *code = malloc(n + 1);
    if (!R || !code) {
        free(R);
        free(code);
        return -1;
    }
    memcpy(R, W, n * OR_V * sizeof(float));
    for (int s = 0; s < OR_STAGES; ++s) {
        err[s] = rvq_apply_stage(n, R, cb + (size_t)s * OR_K * OR_V, code);
        rvq_scatter_codes(rows, nv, s, code, codes);
    }
    free(R);
    free(code);
    return 0;
}
