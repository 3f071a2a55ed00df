/*
 * AirCache oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded fp64 CPU restatement of AirCache's one-shot
 * post-prefill visual KV-cache compression.  Only the test-suite, the smoke
 * check and the CPU-baseline leg of the benchmark may load this library; the
 * product (the CUDA library under lvlm_kv_cache_gb300/) never does, and the two
 * share no code, header, table or helper.
 *
 * Source of every formula: the paper-notes page "AirCache: Activating
 * Inter-Modal Relevancy KV Cache Compression for Efficient Large
 * Vision-Language Model Inference" (ICCV 2025), section "Method details":
 *   - "Key design 1: Elite Observation Window": the prompt layout
 *     X = Concat(X_v, X_t), the text self-attention Att, the elite set k,
 *     the cross-modal attention A_vtk and the visual importance I_v;
 *   - "Key design 2: Layer-wise KV Cache Budget Allocation": strength s_t,
 *     skewness s_k and the layer budget r_hat = 1/2 (s'_t + s'_k) r;
 *   - "Loss / training strategy": the one-shot schedule (save every layer,
 *     then budget all layers, then compress).
 *
 * Readings of points the page leaves open (each is listed in the design notes):
 *   R1  scores are computed per query head and averaged over all H_q heads;
 *       the elite set is taken on the head-mean softmax row P; query head h
 *       reads KV head floor(h / (H_q/H_kv)); one visual index set per layer.
 *   R2  D under the square root is the head dimension.
 *   R3  A_vtk carries no causal mask.
 *   R5  sigma in s_k is the sample standard deviation (n-1); sigma == 0
 *       gives s_k = 0.
 *   R6  s'_t = s_t / mean_l s_t and s'_k = (s_k - min_l s_k + 1e-6) /
 *       mean_l(s_k - min_l s_k + 1e-6), per request over its own layers;
 *       if mean_l s_t == 0 every s'_t is 1.
 *   R7  keep_l = clamp(floor(r_l * N_v + 1/2), 1, N_v).
 *   R8  top-k by I_v, ties to the lower index, output in ascending order.
 *   R9  the elite threshold is inclusive (>=).
 *   R10 every text token is kept in every layer, after the kept visual rows.
 *   R14 the ablation windows of the same page (section "Ablation studies",
 *       observation-window table): a continuous window of w = 16 or 32 is the
 *       last w text tokens, "all text tokens" is every text token; either set
 *       takes the elite set's place (its queries score, its keys join the
 *       softmax).  The visual window of 32 is the last 32 visual tokens (all of
 *       them if fewer): their queries attend over the visual keys only (the
 *       window's own keys are visual keys already), and the visual columns
 *       averaged over the window rows and the query heads give I_v; it reads
 *       the visual tokens' queries.
 *   R15 the ablation budgets (same section, layer-budget table): uniform
 *       r_l = r; PyramidKV-style, linear in depth from (2 - 1/beta) r at layer
 *       0 to r / beta at the last layer (mean r; beta = 20, PyramidKV's
 *       default, the page gives none); strength only r_l = s'_t r; skewness
 *       only r_l = s'_k r; keep_l as in R7.
 *   R16 a decode step (the consumer of the compacted cache) is plain softmax
 *       attention of the step's query over every cached row, per query head,
 *       with the head map of R1 and no mask.
 *   R18 a visual span at an offset (the multimodal-layout page, section on
 *       the correct sequence layout: system text, then the visual tokens, then
 *       the question): request b's prompt is [n_p prefix text][n_v visual]
 *       [suffix text]; "text" is every non-visual token, prefix then suffix,
 *       and text index j is prompt row j (j < n_p) or n_v + j (j >= n_p);
 *       visual index i is prompt row n_p + i.  Every step above runs in those
 *       indices unchanged (the last text query is the prompt's last token);
 *       compaction writes the kept visual rows, then the text rows in text
 *       order.  n_p = 0 is the layout X = Concat(X_v, X_t).
 *   R19 one index set per KV head (the edge-device compression page: group-wise
 *       top-k, one decision per KV group): I_v^(h) averages the visual columns
 *       over the g query heads of KV group h and the elite rows, so that
 *       mean_h I_v^(h) = I_v; the layer's budget keep_l stays the one of I_v;
 *       KV head h keeps the keep_l visual positions with the largest I_v^(h)
 *       (R8's tie and order rules), and its compacted rows are those
 *       positions, then every text row.
 *   R17 int8 storage of the kept cache (LLM KV-compression notes, section
 *       "Quantization stacked on compression": quantise after the token
 *       compression, one scale per head = the head's largest |value| over the
 *       quantisation range; KV-cache tutorial page, section "Quantization":
 *       symmetric q = clip(round(x/s), q_min, q_max), x_hat = s q).  Per
 *       compacted unit (layer, request), per KV head, K and V separately:
 *       s = max|x| / 127 over the unit's rows and the head's D values,
 *       q = clip(round(x / s), -127, 127) with round half away from zero;
 *       s and x / s are evaluated in fp32 (the precision that decides the
 *       integer code on the device too); an all-zero head has s = 0, q = 0.
 *
 * Element access: tensors are token-major [tokens][heads][D] with explicit
 * element strides for the token and head axes and D contiguous; the element
 * type is fp32 or bf16 (decoded here, exactly, by a 16-bit shift).
 */
#include "aircache_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- access */

static double elem(const oracle_view* t, int64_t tok, int64_t head, int64_t i) {
    int64_t off = tok * t->stride_tok + head * t->stride_head + i;
    if (t->dtype == ORACLE_F32) {
        return (double)((const float*)t->base)[off];
    }
    uint16_t bits = ((const uint16_t*)t->base)[off];
    uint32_t word = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

/* Prompt rows of visual index i and text index j (R18). */
static int64_t vis_row(int n_p, int i) { return (int64_t)n_p + i; }
static int64_t text_row(int n_p, int n_v, int j) { return j < n_p ? (int64_t)j : (int64_t)n_v + j; }

/* q_row . k_row / sqrt(D), both rows read in fp64 (R2: D = head dimension). */
static double scaled_dot(const oracle_view* q, int64_t q_tok, int64_t q_head,
                         const oracle_view* k, int64_t k_tok, int64_t k_head, int d) {
    double s = 0.0;
    for (int i = 0; i < d; ++i) {
        s += elem(q, q_tok, q_head, i) * elem(k, k_tok, k_head, i);
    }
    return s / sqrt((double)d);
}

/* ------------------------------------------------------- elite window */

/*
 * "Key design 1", Att equation and elite set k.
 * Att = Softmax(Q_t K_t^T / sqrt(D)); only its last row (the last text query
 * against every text key) is needed.  Per R1 the row is formed per query head
 * and averaged over heads: P[j] = (1/H_q) sum_h softmax_j(q_h[N_t-1] . k[N_v+j]).
 * The elite set is {j : P[j] >= alpha * max P} in ascending order (R9).
 *
 * q      : text queries of this request, row t = text token t (0..N_t-1).
 * k      : keys of this request, row c = prompt position c (visual 0..N_v-1,
 *          then text N_v..N_v+N_t-1) -- the layout X = Concat(X_v, X_t).
 * p_out  : [n_t] the head-mean row P (may be NULL).
 * elite  : [n_t] receives the elite positions (text-relative, ascending).
 * returns N_tk, or -1 on bad arguments.
 */
int oracle_elite(const oracle_view* q, const oracle_view* k, int h_q, int h_kv, int d,
                 int n_v, int n_t, int n_p, double alpha, double* p_out, int32_t* elite) {
    if (h_q <= 0 || h_kv <= 0 || h_q % h_kv != 0 || n_t <= 0 || d <= 0 || n_p < 0 || n_p > n_t) return -1;
    const int g = h_q / h_kv;
    double* logit = (double*)malloc(sizeof(double) * (size_t)n_t);
    double* P = (double*)calloc((size_t)n_t, sizeof(double));
    if (!logit || !P) { free(logit); free(P); return -1; }

    for (int h = 0; h < h_q; ++h) {
        const int kvh = h / g;
        double m = -INFINITY;
        for (int j = 0; j < n_t; ++j) {
            logit[j] = scaled_dot(q, n_t - 1, h, k, text_row(n_p, n_v, j), kvh, d);
            if (logit[j] > m) m = logit[j];
        }
        double z = 0.0;
        for (int j = 0; j < n_t; ++j) z += exp(logit[j] - m);
        for (int j = 0; j < n_t; ++j) P[j] += exp(logit[j] - m) / z;
    }
    double mx = -INFINITY;
    for (int j = 0; j < n_t; ++j) {
        P[j] /= (double)h_q;
        if (P[j] > mx) mx = P[j];
    }
    int n_tk = 0;
    for (int j = 0; j < n_t; ++j) {
        if (P[j] >= alpha * mx) elite[n_tk++] = j;
    }
    if (p_out) memcpy(p_out, P, sizeof(double) * (size_t)n_t);
    free(logit);
    free(P);
    return n_tk;
}

/* ------------------------------------------------- cross-modal scoring */

/*
 * "Key design 1", A_vtk and I_v equations.
 * For each query head h and each elite text row e, a softmax over the keys
 * {visual 0..N_v-1} U {text N_v+e' : e' in elite} (no mask, R3); then
 * I_v[i] = 1/(H_q N_tk) sum_h sum_e A_vtk[h, e, i] for i < N_v (R1).
 *
 * iv          : [n_v] output.
 * elite_mass  : [h_q * n_tk] optional output, the softmax mass each row puts on
 *               the elite text keys (index h * n_tk + e).
 * returns 0, or -1 on bad arguments.
 */
int oracle_score(const oracle_view* q, const oracle_view* k, int h_q, int h_kv, int d,
                 int n_v, int n_t, int n_p, const int32_t* elite, int n_tk,
                 double* iv, double* elite_mass, double* iv_heads) {
    if (h_q <= 0 || h_kv <= 0 || h_q % h_kv != 0 || n_v <= 0 || n_tk <= 0 || n_p < 0 || n_p > n_t) return -1;
    for (int e = 0; e < n_tk; ++e) {
        if (elite[e] < 0 || elite[e] >= n_t) return -1;
    }
    const int g = h_q / h_kv;
    const int n_keys = n_v + n_tk;
    double* logit = (double*)malloc(sizeof(double) * (size_t)n_keys);
    if (!logit) return -1;
    for (int i = 0; i < n_v; ++i) iv[i] = 0.0;
    if (iv_heads) for (int64_t i = 0; i < (int64_t)h_kv * n_v; ++i) iv_heads[i] = 0.0;

    for (int h = 0; h < h_q; ++h) {
        const int kvh = h / g;
        for (int e = 0; e < n_tk; ++e) {
            const int64_t q_tok = elite[e];
            double m = -INFINITY;
            for (int c = 0; c < n_v; ++c) {
                logit[c] = scaled_dot(q, q_tok, h, k, vis_row(n_p, c), kvh, d);
                if (logit[c] > m) m = logit[c];
            }
            for (int e2 = 0; e2 < n_tk; ++e2) {
                logit[n_v + e2] = scaled_dot(q, q_tok, h, k, text_row(n_p, n_v, elite[e2]), kvh, d);
                if (logit[n_v + e2] > m) m = logit[n_v + e2];
            }
            double z = 0.0;
            for (int c = 0; c < n_keys; ++c) z += exp(logit[c] - m);
            for (int c = 0; c < n_v; ++c) iv[c] += exp(logit[c] - m) / z;
            if (iv_heads)
                for (int c = 0; c < n_v; ++c) iv_heads[(int64_t)kvh * n_v + c] += exp(logit[c] - m) / z;
            if (elite_mass) {
                double mass = 0.0;
                for (int e2 = 0; e2 < n_tk; ++e2) mass += exp(logit[n_v + e2] - m) / z;
                elite_mass[(int64_t)h * n_tk + e] = mass;
            }
        }
    }
    const double norm = (double)h_q * (double)n_tk;
    for (int i = 0; i < n_v; ++i) iv[i] /= norm;
    if (iv_heads) {
        const double norm_h = (double)g * (double)n_tk;  /* R19: a group's g query heads */
        for (int64_t i = 0; i < (int64_t)h_kv * n_v; ++i) iv_heads[i] /= norm_h;
    }
    free(logit);
    return 0;
}

/* ------------------------------------------------ strength and skewness */

/*
 * "Key design 2", strength s_t = sum_i I_v[i] and skewness
 * s_k = N_v / ((N_v-1)(N_v-2)) sum_i ((I_v[i] - mu) / sigma)^3, with sigma the
 * sample standard deviation (R5).  Needs N_v >= 3.
 * out[0] = s_t, out[1] = s_k, out[2] = mu, out[3] = sigma.
 */
int oracle_stats(const double* iv, int n_v, double* out) {
    if (n_v < 3) return -1;
    double s_t = 0.0;
    for (int i = 0; i < n_v; ++i) s_t += iv[i];
    const double mu = s_t / n_v;
    double ss = 0.0;
    for (int i = 0; i < n_v; ++i) ss += (iv[i] - mu) * (iv[i] - mu);
    const double sigma = sqrt(ss / (n_v - 1));
    double s_k = 0.0;
    if (sigma > 0.0) {
        double cube = 0.0;
        for (int i = 0; i < n_v; ++i) {
            const double z = (iv[i] - mu) / sigma;
            cube += z * z * z;
        }
        s_k = (double)n_v / ((double)(n_v - 1) * (double)(n_v - 2)) * cube;
    }
    out[0] = s_t;
    out[1] = s_k;
    out[2] = mu;
    out[3] = sigma;
    return 0;
}

/* ------------------------------------------------------- layer budget */

/*
 * R6: s'_t[l] = s_t[l] / mean s_t (1 if the mean is 0) and
 * s'_k[l] = (s_k[l] - min s_k + 1e-6) / mean(s_k - min s_k + 1e-6).
 */
static void normalised_layers(const double* s_t, const double* s_k, int n_layers, double* st_n,
                              double* sk_n) {
    double mean_st = 0.0, min_sk = INFINITY;
    for (int l = 0; l < n_layers; ++l) {
        mean_st += s_t[l];
        if (s_k[l] < min_sk) min_sk = s_k[l];
    }
    mean_st /= n_layers;
    double mean_u = 0.0;
    for (int l = 0; l < n_layers; ++l) mean_u += s_k[l] - min_sk + 1e-6;
    mean_u /= n_layers;
    for (int l = 0; l < n_layers; ++l) {
        st_n[l] = (mean_st != 0.0) ? s_t[l] / mean_st : 1.0;
        sk_n[l] = (s_k[l] - min_sk + 1e-6) / mean_u;
    }
}

/* R7: keep = clamp(floor(r_l N_v + 1/2), 1, N_v). */
static int32_t keep_of(double rl, int n_v) {
    double kf = floor(rl * (double)n_v + 0.5);
    if (kf < 1.0) kf = 1.0;
    if (kf > (double)n_v) kf = (double)n_v;
    return (int32_t)kf;
}

/*
 * "Key design 2", budget r_hat = 1/2 (s'_t + s'_k) r with the cross-layer
 * normalisation of R6, over the n_layers layers of one request, then the keep
 * count of R7.
 * s_t, s_k : [n_layers]; r_l : [n_layers] output (may be NULL);
 * keep : [n_layers] output.
 */
int oracle_budget(const double* s_t, const double* s_k, int n_layers, int n_v, double r,
                  double* r_l, int32_t* keep) {
    if (n_layers <= 0 || n_v <= 0) return -1;
    double* st_n = (double*)malloc(sizeof(double) * (size_t)n_layers);
    double* sk_n = (double*)malloc(sizeof(double) * (size_t)n_layers);
    if (!st_n || !sk_n) { free(st_n); free(sk_n); return -1; }
    normalised_layers(s_t, s_k, n_layers, st_n, sk_n);
    for (int l = 0; l < n_layers; ++l) {
        const double rl = 0.5 * (st_n[l] + sk_n[l]) * r;
        keep[l] = keep_of(rl, n_v);
        if (r_l) r_l[l] = rl;
    }
    free(st_n);
    free(sk_n);
    return 0;
}

/* ----------------------------------------------------- ablation variants */

/*
 * "Ablation studies", observation-window table (R14): the window that replaces
 * the elite set.  mode 1: last 16 text tokens; 2: last 32; 3: every text token.
 * positions : [n_t] receives the window (text-relative, ascending).
 * returns its size, or -1 for an unknown mode or n_t < 1.
 */
int oracle_window(int n_t, int mode, int32_t* positions) {
    if (n_t < 1) return -1;
    int w;
    if (mode == 1) w = 16;
    else if (mode == 2) w = 32;
    else if (mode == 3) w = n_t;
    else return -1;
    if (w > n_t) w = n_t;
    for (int e = 0; e < w; ++e) positions[e] = n_t - w + e;
    return w;
}

/* R14's visual window: the last min(32, n_v) visual indices, ascending. */
int oracle_window_visual(int n_v, int32_t* positions) {
    if (n_v < 1) return -1;
    const int w = n_v < 32 ? n_v : 32;
    for (int e = 0; e < w; ++e) positions[e] = n_v - w + e;
    return w;
}

/*
 * I_v of one (request, layer) for R14's visual window: qv holds the request's
 * visual-token queries (row i = visual index i), k its keys in prompt order
 * (R18); window rows pos[0..n_w), softmax over the n_v visual keys only.
 */
int oracle_score_visual_window(const oracle_view* qv, const oracle_view* k, int h_q, int h_kv, int d, int n_v,
                               int n_p, const int32_t* pos, int n_w, double* iv) {
    if (h_q <= 0 || h_kv <= 0 || h_q % h_kv != 0 || n_v <= 0 || n_w <= 0 || n_p < 0) return -1;
    for (int e = 0; e < n_w; ++e) if (pos[e] < 0 || pos[e] >= n_v) return -1;
    const int g = h_q / h_kv;
    double* logit = (double*)malloc(sizeof(double) * (size_t)n_v);
    if (!logit) return -1;
    for (int i = 0; i < n_v; ++i) iv[i] = 0.0;
    for (int h = 0; h < h_q; ++h) {
        const int kvh = h / g;
        for (int e = 0; e < n_w; ++e) {
            double m = -INFINITY;
            for (int c = 0; c < n_v; ++c) {
                logit[c] = scaled_dot(qv, pos[e], h, k, vis_row(n_p, c), kvh, d);
                if (logit[c] > m) m = logit[c];
            }
            double z = 0.0;
            for (int c = 0; c < n_v; ++c) z += exp(logit[c] - m);
            for (int c = 0; c < n_v; ++c) iv[c] += exp(logit[c] - m) / z;
        }
    }
    for (int i = 0; i < n_v; ++i) iv[i] /= (double)h_q * (double)n_w;
    free(logit);
    return 0;
}

/*
 * "Ablation studies", layer-budget table (R15): budget mode 0 is the method's
 * own (oracle_budget); 1 uniform; 2 PyramidKV-style (beta = 20); 3 strength
 * only; 4 skewness only.  Arguments as oracle_budget.
 */
int oracle_budget_variant(const double* s_t, const double* s_k, int n_layers, int n_v, double r,
                          int mode, double* r_l, int32_t* keep) {
    if (n_layers <= 0 || n_v <= 0 || mode < 0 || mode > 4) return -1;
    if (mode == 0) return oracle_budget(s_t, s_k, n_layers, n_v, r, r_l, keep);
    double* st_n = (double*)malloc(sizeof(double) * (size_t)n_layers);
    double* sk_n = (double*)malloc(sizeof(double) * (size_t)n_layers);
    if (!st_n || !sk_n) { free(st_n); free(sk_n); return -1; }
    normalised_layers(s_t, s_k, n_layers, st_n, sk_n);
    const double beta = 20.0;
    const double r_top = r / beta;
    const double r_bottom = 2.0 * r - r_top;
    for (int l = 0; l < n_layers; ++l) {
        double rl;
        if (mode == 1) {
            rl = r;
        } else if (mode == 2) {
            const double t = n_layers > 1 ? (double)l / (double)(n_layers - 1) : 0.5;
            rl = r_bottom + (r_top - r_bottom) * t;
        } else if (mode == 3) {
            rl = st_n[l] * r;
        } else {
            rl = sk_n[l] * r;
        }
        keep[l] = keep_of(rl, n_v);
        if (r_l) r_l[l] = rl;
    }
    free(st_n);
    free(sk_n);
    return 0;
}

/* ---------------------------------------------------------- selection */

/* Sort key for the selection: larger I_v first, then lower index (R8). */
typedef struct { double v; int32_t i; } scored_index;

static int by_score_then_index(const void* a, const void* b) {
    const scored_index* x = (const scored_index*)a;
    const scored_index* y = (const scored_index*)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->i > y->i) - (x->i < y->i);
}

static int ascending_int(const void* a, const void* b) {
    const int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/*
 * Keep the `keep` visual positions with the largest I_v (R8): order all
 * positions by (I_v descending, index ascending), take the first `keep`,
 * return them sorted ascending in idx[0..keep).
 */
int oracle_select(const double* iv, int n_v, int keep, int32_t* idx) {
    if (n_v <= 0 || keep < 0 || keep > n_v) return -1;
    scored_index* s = (scored_index*)malloc(sizeof(scored_index) * (size_t)n_v);
    if (!s) return -1;
    for (int i = 0; i < n_v; ++i) { s[i].v = iv[i]; s[i].i = i; }
    qsort(s, (size_t)n_v, sizeof(scored_index), by_score_then_index);
    for (int j = 0; j < keep; ++j) idx[j] = s[j].i;
    qsort(idx, (size_t)keep, sizeof(int32_t), ascending_int);
    free(s);
    return 0;
}

/* -------------------------------------------------------- compaction */

/*
 * "Loss / training strategy" step 3 (the compressed cache feeds decoding) and
 * R10: the compacted rows of one (request, layer) are [K_v[idx]; K_t], i.e. the
 * kept visual positions in ascending order followed by every text position.
 * Rows are copied element by element (bit-exact, in the source type) into a
 * dense [rows][h_kv][d] destination.  Returns the number of rows written.
 */
int64_t oracle_compact(const oracle_view* src, int h_kv, int d, int n_v, int n_t, int n_p,
                       const int32_t* idx, int keep, void* dst) {
    if (n_p < 0 || n_p > n_t) return -1;
    const size_t esize = (src->dtype == ORACLE_F32) ? 4 : 2;
    unsigned char* out = (unsigned char*)dst;
    int64_t row = 0;
    for (int j = 0; j < keep + n_t; ++j) {
        const int64_t tok = (j < keep) ? vis_row(n_p, idx[j]) : text_row(n_p, n_v, j - keep);
        for (int h = 0; h < h_kv; ++h) {
            const unsigned char* from = (const unsigned char*)src->base +
                (size_t)(tok * src->stride_tok + h * src->stride_head) * esize;
            memcpy(out + ((size_t)row * h_kv + h) * d * esize, from, (size_t)d * esize);
        }
        ++row;
    }
    return row;
}

/* ------------------------------------------------------ one request */

/*
 * The one-shot schedule of "Loss / training strategy" for one request over
 * all of its layers: elite + score + stats for every layer, then one budget
 * over the layers, then selection per layer.  Compaction is left to
 * oracle_compact so that callers choose where rows go.
 *
 * q[l], k[l] : views of layer l restricted to this request.
 * iv         : [n_layers * n_v] output; elite: [n_layers * max(n_t, 32)]; n_tk: [n_layers];
 * stats      : [n_layers * 4]; keep: [n_layers]; idx: [n_layers * n_v].
 */
int oracle_request_variant(const oracle_view* q, const oracle_view* k, int n_layers, int h_q,
                           int h_kv, int d, int n_v, int n_t, int n_p, double alpha, double r, int window_mode,
                           int budget_mode, double* iv, int32_t* elite, int32_t* n_tk, double* stats,
                           int32_t* keep, int32_t* idx, double* iv_heads, int32_t* idx_heads,
                           const oracle_view* qv) {
    if (window_mode == 4 && (!qv || iv_heads)) return -1;  /* the visual window reads qv; one set per layer */
    double* s_t = (double*)malloc(sizeof(double) * (size_t)n_layers);
    double* s_k = (double*)malloc(sizeof(double) * (size_t)n_layers);
    if (!s_t || !s_k) { free(s_t); free(s_k); return -1; }
    int rc = 0;
    for (int l = 0; l < n_layers && rc == 0; ++l) {
        int32_t* el = elite + (int64_t)l * (n_t > 32 ? n_t : 32);
        const int ntk = window_mode == 0   ? oracle_elite(&q[l], &k[l], h_q, h_kv, d, n_v, n_t, n_p, alpha, NULL, el)
                        : window_mode == 4 ? oracle_window_visual(n_v, el)
                                           : oracle_window(n_t, window_mode, el);
        if (ntk <= 0) { rc = -1; break; }
        n_tk[l] = ntk;
        double* ivl = iv + (int64_t)l * n_v;
        if (window_mode == 4)
            rc = oracle_score_visual_window(&qv[l], &k[l], h_q, h_kv, d, n_v, n_p, el, ntk, ivl);
        else
            rc = oracle_score(&q[l], &k[l], h_q, h_kv, d, n_v, n_t, n_p, el, ntk, ivl, NULL,
                              iv_heads ? iv_heads + (int64_t)l * h_kv * n_v : NULL);
        if (rc == 0) rc = oracle_stats(ivl, n_v, stats + (int64_t)l * 4);
        if (rc == 0) { s_t[l] = stats[l * 4 + 0]; s_k[l] = stats[l * 4 + 1]; }
    }
    if (rc == 0) rc = oracle_budget_variant(s_t, s_k, n_layers, n_v, r, budget_mode, NULL, keep);
    for (int l = 0; l < n_layers && rc == 0; ++l) {
        rc = oracle_select(iv + (int64_t)l * n_v, n_v, keep[l], idx + (int64_t)l * n_v);
        /* R19: each KV head's own set, with the layer's keep count */
        for (int h = 0; h < h_kv && rc == 0 && iv_heads && idx_heads; ++h) {
            const int64_t o = ((int64_t)l * h_kv + h) * n_v;
            rc = oracle_select(iv_heads + o, n_v, keep[l], idx_heads + o);
        }
    }
    free(s_t);
    free(s_k);
    return rc;
}

/* The method itself: the elite window and the strength + skewness budget. */
int oracle_request(const oracle_view* q, const oracle_view* k, int n_layers, int h_q, int h_kv,
                   int d, int n_v, int n_t, double alpha, double r,
                   double* iv, int32_t* elite, int32_t* n_tk, double* stats,
                   int32_t* keep, int32_t* idx) {
    return oracle_request_variant(q, k, n_layers, h_q, h_kv, d, n_v, n_t, 0, alpha, r, 0, 0, iv, elite,
                                  n_tk, stats, keep, idx, NULL, NULL, NULL);
}

/* ------------------------------------------------------- decode consumer */

/*
 * One decode step over a KV cache (the KV-cache tutorial page, section
 * "Prefill and Decode": each step brings one new query, which reads every
 * cached key and value; the edge-device compression page, head-wise top-k
 * scheme: once the cache is compacted, decoding is plain dense attention over
 * the compacted rows).  R16: for query head h, reading KV head h / (H_q/H_kv)
 * as in R1,
 *   o_h = sum_j softmax_j(q_h . k_j / sqrt(D)) v_j
 * over every row j of the cache, with no mask (every cached row precedes the
 * query).
 *
 * q    : a view whose token 0 is the query, [H_q][D];
 * k, v : views whose tokens 0..n_rows-1 are the cached rows, [H_kv][D] each;
 * out  : [H_q * D] fp64, row h = o_h.
 * returns 0, or -1 on bad arguments (n_rows < 1 among them).
 */
int oracle_decode(const oracle_view* q, const oracle_view* k, const oracle_view* v, int h_q, int h_kv,
                  int d, int64_t n_rows, double* out) {
    if (h_q <= 0 || h_kv <= 0 || h_q % h_kv != 0 || d <= 0 || n_rows < 1) return -1;
    const int group = h_q / h_kv;
    double* w = (double*)malloc(sizeof(double) * (size_t)n_rows);
    if (!w) return -1;
    for (int h = 0; h < h_q; ++h) {
        const int kv_head = h / group;
        /* softmax weights of this head over the rows, max-subtracted */
        double top = -INFINITY;
        for (int64_t j = 0; j < n_rows; ++j) {
            w[j] = scaled_dot(q, 0, h, k, j, kv_head, d);
            top = fmax(top, w[j]);
        }
        double total = 0.0;
        for (int64_t j = 0; j < n_rows; ++j) {
            w[j] = exp(w[j] - top);
            total += w[j];
        }
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int64_t j = 0; j < n_rows; ++j) acc += w[j] / total * elem(v, j, kv_head, i);
            out[(int64_t)h * d + i] = acc;
        }
    }
    free(w);
    return 0;
}

/* ------------------------------------------------------- int8 kept cache */

/* The elementary symmetric step of R17 for one value: clip(round(x / s)),
 * x / s in fp32, half away from zero; s == 0 gives 0. */
int oracle_quant_code(float x, float s) {
    if (s == 0.0f) return 0;
    const float t = x / s;
    float r = roundf(t);
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    return (int)r;
}

/*
 * R17 over one compacted unit: rows 0..n_rows-1 of `src` ([rows][H_kv][D]).
 * codes: [n_rows][h_kv][d] int8, dense; scales: [h_kv] fp32 (s of each head).
 * returns 0, or -1 on bad arguments.
 */
int oracle_quantize_int8(const oracle_view* src, int64_t n_rows, int h_kv, int d, int8_t* codes,
                         float* scales) {
    if (n_rows < 0 || h_kv <= 0 || d <= 0) return -1;
    for (int h = 0; h < h_kv; ++h) {
        float big = 0.0f;
        for (int64_t j = 0; j < n_rows; ++j)
            for (int i = 0; i < d; ++i) {
                const float a = fabsf((float)elem(src, j, h, i));
                if (a > big) big = a;
            }
        const float s = big / 127.0f;
        scales[h] = s;
        for (int64_t j = 0; j < n_rows; ++j)
            for (int i = 0; i < d; ++i)
                codes[(j * h_kv + h) * d + i] = (int8_t)oracle_quant_code((float)elem(src, j, h, i), s);
    }
    return 0;
}

/*
 * R19 compaction with one index set per KV head: row j of head h is visual
 * position idx_heads[h * n_v + j] (j < keep) or text index j - keep, in the
 * prompt layout of R18.  dst: dense [keep + n_t][h_kv][d].  Returns the rows.
 */
int64_t oracle_compact_heads(const oracle_view* src, int h_kv, int d, int n_v, int n_t, int n_p,
                             const int32_t* idx_heads, int keep, void* dst) {
    if (n_p < 0 || n_p > n_t) return -1;
    const size_t esize = (src->dtype == ORACLE_F32) ? 4 : 2;
    unsigned char* out = (unsigned char*)dst;
    for (int j = 0; j < keep + n_t; ++j) {
        for (int h = 0; h < h_kv; ++h) {
            const int64_t tok = (j < keep) ? vis_row(n_p, idx_heads[(int64_t)h * n_v + j]) : text_row(n_p, n_v, j - keep);
            const unsigned char* from = (const unsigned char*)src->base +
                (size_t)(tok * src->stride_tok + h * src->stride_head) * esize;
            memcpy(out + ((size_t)j * h_kv + h) * d * esize, from, (size_t)d * esize);
        }
    }
    return (int64_t)keep + n_t;
}
