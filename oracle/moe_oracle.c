/*
 * moe_oracle.c -- plain, slow CPU oracle of the sparse Mixture-of-Experts block
 * (Qwen3-MoE style: router, softmax over experts, top-k, renormalisation,
 * grouped SwiGLU experts, weighted combine).
 *
 * TEST INFRASTRUCTURE.  Only the test-suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or helper with the CUDA library, and neither one includes or links the
 * other.  Inputs are widened exactly (fp32 -> double, bf16 -> double, 4-bit
 * code -> codebook[code] * scale in double) and every step runs in double.
 *
 * Sources.  The op sequence is the one the unsloth commit page 80aaf1121b
 * ("Qwen3-30B-A3B decode ... CUDA-graph capture", paragraph on the grouped_mm
 * backend) names for the MoE block: expert histogram (bincount, later a
 * capture-safe scatter_add_), cumsum, argsort, torch._grouped_mm, index_add_.
 * The pages name those ops but print no formulas, so each step below is the
 * plain definition of what the op computes in a Qwen3-MoE sparse block:
 *
 *   A  logits[t,e] = sum_h x[t,h] * Wr[e,h] (+ b[e] when a router bias is given)
 *   B  p[t,:] = softmax over all E logits (max-subtracted);
 *      S_t = the k experts with the largest logits, largest first; equal
 *      logits put the lower expert index first;
 *      w[t,j] = p[S_j] / sum_{i<k} p[S_i] when norm_topk, else p[S_j];
 *      tie_margin[t] = logit(S_{k-1}) - logit of the (k+1)-th choice
 *      (+inf when k == E).  The unsloth commit page cc4832b605 (parity
 *      paragraph) attributes its only divergences to top-k ties, which is
 *      why the margin is reported.
 *   C  counts[e] = #{a : ids[a] == e} over the A = T*k assignments a = t*k + j;
 *      offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e]
 *   D  order[p] = the p-th assignment when sorted by (expert id, a), i.e. a
 *      stable sort by expert; pos[order[p]] = p
 *   E  for permuted row p of expert e, source token t = order[p] / k:
 *      g = x_t . Wg[e]^T, u = x_t . Wu[e]^T, h = SiLU(g) * u,
 *      SiLU(z) = z / (1 + exp(-z))
 *   F  y[p] = h . Wd[e]^T
 *   G  out[t] = sum_{j<k} w[t,j] * y[pos[t*k + j]], summed in j order
 *
 * 4-bit weights: element (e, r, c) of a [rows][cols] matrix sits in byte
 * ((e*rows + r)*cols + c) / 2, low nibble for even c and high nibble for odd c;
 * its value is codebook[code] * scale[e, r, c / q_block], scale a bf16 value.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared moe_oracle.c -lm
 * (no FMA contraction, so x86_64 and aarch64 hosts round identically).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_Q4 = 2 };

/* One stack of E expert matrices, each [rows][cols] row-major, cols = input dim. */
typedef struct {
    int32_t dtype;
    int32_t q_block;
    int64_t rows;
    int64_t cols;
    const void *data;         /* float, bf16 bits (uint16) or packed codes (uint8) */
    const uint16_t *scales;   /* 4-bit only: bf16 bits [E][rows][cols / q_block] */
    const float *codebook;    /* 4-bit only: 16 entries */
} orc_matrix;

static double widen_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Element i of an activation-dtype array (fp32 or bf16 bits). */
static double act_at(int dtype, const void *p, int64_t i)
{
    if (dtype == ORC_F32) return (double)((const float *)p)[i];
    return widen_bf16(((const uint16_t *)p)[i]);
}

static double weight_at(const orc_matrix *m, int64_t e, int64_t r, int64_t c)
{
    int64_t idx = (e * m->rows + r) * m->cols + c;
    if (m->dtype == ORC_F32) return (double)((const float *)m->data)[idx];
    if (m->dtype == ORC_BF16) return widen_bf16(((const uint16_t *)m->data)[idx]);
    {
        uint8_t byte = ((const uint8_t *)m->data)[idx / 2];
        int code = (idx & 1) ? (byte >> 4) : (byte & 0x0F);
        int64_t nblk = m->cols / m->q_block;
        double scale = widen_bf16(m->scales[(e * m->rows + r) * nblk + c / m->q_block]);
        return (double)m->codebook[code] * scale;
    }
}

static int check_matrix(const orc_matrix *m, int64_t rows, int64_t cols)
{
    if (!m || !m->data || m->rows != rows || m->cols != cols) return -1;
    if (m->dtype == ORC_Q4) {
        if (!m->scales || !m->codebook || m->q_block <= 0 || cols % m->q_block || cols % 2) return -1;
    } else if (m->dtype != ORC_F32 && m->dtype != ORC_BF16) {
        return -1;
    }
    return 0;
}

static size_t act_size(int dtype) { return dtype == ORC_F32 ? 4 : 2; }

/* Step A for tokens [0, T): logits[t*E + e]. */
int orc_router_logits(int T, int H, int E, int act_dtype, const void *x, const void *w_router,
                      const float *bias, double *logits)
{
    if (T < 0 || H <= 0 || E <= 0 || !x || !w_router || !logits) return -1;
    if (act_dtype != ORC_F32 && act_dtype != ORC_BF16) return -1;
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double s = 0.0;
            for (int h = 0; h < H; ++h)
                s += act_at(act_dtype, x, (int64_t)t * H + h) * act_at(act_dtype, w_router, (int64_t)e * H + h);
            if (bias) s += (double)bias[e];
            logits[(int64_t)t * E + e] = s;
        }
    }
    return 0;
}

/* Step B for tokens [0, T). */
int orc_select_topk(int T, int E, int k, int norm_topk, const double *logits, int32_t *ids,
                    double *weights, double *tie_margin)
{
    if (T < 0 || E <= 0 || k <= 0 || k > E || !logits || !ids || !weights) return -1;
    int *rank = (int *)malloc(sizeof(int) * (size_t)E);
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    if (!rank || !p) { free(rank); free(p); return -2; }
    for (int t = 0; t < T; ++t) {
        const double *l = logits + (int64_t)t * E;
        /* softmax over all experts */
        double m = l[0];
        for (int e = 1; e < E; ++e) if (l[e] > m) m = l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) { p[e] = exp(l[e] - m); z += p[e]; }
        for (int e = 0; e < E; ++e) p[e] /= z;
        /* all experts ordered by logit, largest first; insertion sort is stable,
         * so equal logits keep ascending expert index */
        for (int e = 0; e < E; ++e) rank[e] = e;
        for (int i = 1; i < E; ++i) {
            int v = rank[i];
            int j = i - 1;
            while (j >= 0 && l[rank[j]] < l[v]) { rank[j + 1] = rank[j]; --j; }
            rank[j + 1] = v;
        }
        double psum = 0.0;
        for (int j = 0; j < k; ++j) psum += p[rank[j]];
        for (int j = 0; j < k; ++j) {
            ids[(int64_t)t * k + j] = rank[j];
            weights[(int64_t)t * k + j] = norm_topk ? p[rank[j]] / psum : p[rank[j]];
        }
        if (tie_margin) tie_margin[t] = (k < E) ? l[rank[k - 1]] - l[rank[k]] : INFINITY;
    }
    free(rank);
    free(p);
    return 0;
}

/* Steps C and D: counting sort of the A assignments by expert id. */
int orc_permute(int A, int E, const int32_t *ids, int32_t *counts, int32_t *offsets,
                int32_t *order, int32_t *pos)
{
    if (A < 0 || E <= 0 || !counts || !offsets || (A > 0 && (!ids || !order || !pos))) return -1;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int a = 0; a < A; ++a) {
        if (ids[a] < 0 || ids[a] >= E) return -3;
        counts[ids[a]] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    /* scanning a upward and appending to each expert's segment keeps a ascending */
    int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    if (!fill) return -2;
    for (int e = 0; e < E; ++e) fill[e] = offsets[e];
    for (int a = 0; a < A; ++a) {
        int p = fill[ids[a]]++;
        order[p] = a;
        pos[a] = p;
    }
    free(fill);
    return 0;
}

/*
 * LoRA adapters on the experts: rank r, fp32, one (A, B) pair per expert and
 * projection, adding scale * B A to the projection's weight:
 *   W'_P[e] = W_P[e] + scale * B_P[e] A_P[e],  A_P [E][r][in], B_P [E][out][r],
 * i.e. z = x . W_P[e]^T + scale * (x . A_P[e]^T) . B_P[e]^T.  The unsloth commit page
 * 4f2bfe7f69 benchmarks the model with a rank-16 LoRA on 4-bit weights and names
 * "4bit forward, fp32 LoRA injection" as the inference form; it gives no placement,
 * so the adapters sit on the three expert projections (gate, up, down).
 */
typedef struct {
    int32_t rank;
    double scale;
    const float *a_gate, *b_gate, *a_up, *b_up, *a_down, *b_down;
} orc_lora;

/* scale * sum_q B[e][row][q] * v[q] */
static double lora_out(const orc_lora *l, const float *B, int e, int64_t rows, int64_t row, const double *v)
{
    double s = 0.0;
    for (int q = 0; q < l->rank; ++q) s += (double)B[((int64_t)e * rows + row) * l->rank + q] * v[q];
    return l->scale * s;
}

/* v[q] = sum_c A[e][q][c] * x[c] */
static void lora_in(const orc_lora *l, const float *A, int e, int64_t cols, const double *x, double *v)
{
    for (int q = 0; q < l->rank; ++q) {
        double s = 0.0;
        for (int64_t c = 0; c < cols; ++c) s += (double)A[((int64_t)e * l->rank + q) * cols + c] * x[c];
        v[q] = s;
    }
}

/* Steps E and F for one activation row and one expert, with optional adapters. */
static int expert_mlp(int H, int I, const double *xrow, int e, const orc_matrix *w_gate, const orc_matrix *w_up,
                      const orc_matrix *w_down, const orc_lora *lora, double *h, double *y)
{
    if (H <= 0 || I <= 0 || !xrow || !y || e < 0) return -1;
    if (check_matrix(w_gate, I, H) || check_matrix(w_up, I, H) || check_matrix(w_down, H, I)) return -1;
    if (lora && (lora->rank < 1 || lora->rank > 64 || !lora->a_gate || !lora->b_gate || !lora->a_up ||
                 !lora->b_up || !lora->a_down || !lora->b_down))
        return -1;
    double *hh = h ? h : (double *)malloc(sizeof(double) * (size_t)I);
    if (!hh) return -2;
    double xg[64], xu[64], hd[64];
    if (lora) {
        lora_in(lora, lora->a_gate, e, H, xrow, xg);
        lora_in(lora, lora->a_up, e, H, xrow, xu);
    }
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
            g += xrow[c] * weight_at(w_gate, e, i, c);
            u += xrow[c] * weight_at(w_up, e, i, c);
        }
        if (lora) {
            g += lora_out(lora, lora->b_gate, e, I, i, xg);
            u += lora_out(lora, lora->b_up, e, I, i, xu);
        }
        hh[i] = (g / (1.0 + exp(-g))) * u;
    }
    if (lora) lora_in(lora, lora->a_down, e, I, hh, hd);
    for (int r = 0; r < H; ++r) {
        double s = 0.0;
        for (int i = 0; i < I; ++i) s += hh[i] * weight_at(w_down, e, r, i);
        if (lora) s += lora_out(lora, lora->b_down, e, H, r, hd);
        y[r] = s;
    }
    if (!h) free(hh);
    return 0;
}

/* Steps E and F for one activation row and one expert. h may be NULL. */
int orc_expert_mlp(int H, int I, const double *xrow, int e, const orc_matrix *w_gate,
                   const orc_matrix *w_up, const orc_matrix *w_down, double *h, double *y)
{
    return expert_mlp(H, I, xrow, e, w_gate, w_up, w_down, NULL, h, y);
}

static void widen_row(int act_dtype, const void *x, int64_t t, int H, double *row)
{
    for (int c = 0; c < H; ++c) row[c] = act_at(act_dtype, x, t * H + c);
}

/* Steps E and F over the permuted rows: y[p] for p in [0, T*k). */
int orc_grouped_swiglu(int T, int H, int E, int k, int I, int act_dtype, const void *x,
                       const int32_t *offsets, const int32_t *order, const orc_matrix *w_gate,
                       const orc_matrix *w_up, const orc_matrix *w_down, double *h, double *y)
{
    if (T < 0 || k <= 0 || !x || !offsets || !order || !y) return -1;
    double *row = (double *)malloc(sizeof(double) * (size_t)H);
    if (!row) return -2;
    int rc = 0;
    for (int e = 0; e < E && rc == 0; ++e) {
        for (int p = offsets[e]; p < offsets[e + 1]; ++p) {
            widen_row(act_dtype, x, order[p] / k, H, row);
            rc = orc_expert_mlp(H, I, row, e, w_gate, w_up, w_down,
                                h ? h + (int64_t)p * I : NULL, y + (int64_t)p * H);
            if (rc) break;
        }
    }
    free(row);
    return rc;
}

/* Step G. */
int orc_unpermute(int T, int k, int H, const double *y, const double *weights, const int32_t *pos,
                  double *out)
{
    if (T < 0 || k <= 0 || H <= 0 || !y || !weights || !pos || !out) return -1;
    for (int t = 0; t < T; ++t) {
        for (int c = 0; c < H; ++c) {
            double s = 0.0;
            for (int j = 0; j < k; ++j)
                s += weights[(int64_t)t * k + j] * y[(int64_t)pos[(int64_t)t * k + j] * H + c];
            out[(int64_t)t * H + c] = s;
        }
    }
    return 0;
}

/* Steps A..G over all T tokens, in the order above.  Every intermediate is an output. */
int orc_forward(int T, int H, int E, int k, int I, int norm_topk, int act_dtype, const void *x,
                const void *w_router, const float *bias, const orc_matrix *w_gate,
                const orc_matrix *w_up, const orc_matrix *w_down, double *logits, int32_t *ids,
                double *weights, double *tie_margin, int32_t *counts, int32_t *offsets,
                int32_t *order, int32_t *pos, double *h, double *y, double *out)
{
    int rc = orc_router_logits(T, H, E, act_dtype, x, w_router, bias, logits);
    if (!rc) rc = orc_select_topk(T, E, k, norm_topk, logits, ids, weights, tie_margin);
    if (!rc) rc = orc_permute(T * k, E, ids, counts, offsets, order, pos);
    if (!rc) rc = orc_grouped_swiglu(T, H, E, k, I, act_dtype, x, offsets, order, w_gate, w_up, w_down, h, y);
    if (!rc) rc = orc_unpermute(T, k, H, y, weights, pos, out);
    return rc;
}

/*
 * The block's output for a list of tokens, one token at a time.  out[t] depends
 * only on token t (its own routing and its own k expert rows), so this is the
 * same definition evaluated for a sample of tokens of a large batch.
 */
static int forward_tokens(int ntok, const int32_t *tokens, int H, int E, int k, int I, int norm_topk,
                          int act_dtype, const void *x, const void *w_router, const float *bias,
                          const orc_matrix *w_gate, const orc_matrix *w_up, const orc_matrix *w_down,
                          const orc_lora *lora, int32_t *ids, double *weights, double *tie_margin, double *out)
{
    if (ntok < 0 || !tokens || !x || !out || !ids || !weights) return -1;
    double *logit = (double *)malloc(sizeof(double) * (size_t)E);
    double *row = (double *)malloc(sizeof(double) * (size_t)H);
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    int rc = (logit && row && y) ? 0 : -2;
    size_t es = act_size(act_dtype);
    for (int n = 0; n < ntok && rc == 0; ++n) {
        int64_t t = tokens[n];
        const void *xt = (const char *)x + (size_t)t * (size_t)H * es;
        rc = orc_router_logits(1, H, E, act_dtype, xt, w_router, bias, logit);
        if (!rc) rc = orc_select_topk(1, E, k, norm_topk, logit, ids + (int64_t)n * k,
                                      weights + (int64_t)n * k, tie_margin ? tie_margin + n : NULL);
        if (rc) break;
        widen_row(act_dtype, x, t, H, row);
        double *o = out + (int64_t)n * H;
        for (int c = 0; c < H; ++c) o[c] = 0.0;
        for (int j = 0; j < k && rc == 0; ++j) {
            rc = expert_mlp(H, I, row, ids[(int64_t)n * k + j], w_gate, w_up, w_down, lora, NULL, y);
            for (int c = 0; c < H && rc == 0; ++c) o[c] += weights[(int64_t)n * k + j] * y[c];
        }
    }
    free(logit); free(row); free(y);
    return rc;
}

int orc_forward_tokens(int ntok, const int32_t *tokens, int H, int E, int k, int I, int norm_topk,
                       int act_dtype, const void *x, const void *w_router, const float *bias,
                       const orc_matrix *w_gate, const orc_matrix *w_up, const orc_matrix *w_down,
                       int32_t *ids, double *weights, double *tie_margin, double *out)
{
    return forward_tokens(ntok, tokens, H, E, k, I, norm_topk, act_dtype, x, w_router, bias, w_gate, w_up, w_down,
                          NULL, ids, weights, tie_margin, out);
}

/* orc_forward_tokens with LoRA adapters on the experts. */
int orc_forward_tokens_lora(int ntok, const int32_t *tokens, int H, int E, int k, int I, int norm_topk,
                            int act_dtype, const void *x, const void *w_router, const float *bias,
                            const orc_matrix *w_gate, const orc_matrix *w_up, const orc_matrix *w_down,
                            const orc_lora *lora, int32_t *ids, double *weights, double *tie_margin, double *out)
{
    if (!lora) return -1;
    return forward_tokens(ntok, tokens, H, E, k, I, norm_topk, act_dtype, x, w_router, bias, w_gate, w_up, w_down,
                          lora, ids, weights, tie_margin, out);
}

/*
 * Dense brute force: every token through every expert, then a mask m[t,e]
 * that is w[t,j] on the selected experts and 0 elsewhere:
 *   out[t] = sum_e m[t,e] * expert_e(x_t).
 * Equal to the sparse result by construction of the dispatch; used to check it.
 */
int orc_forward_dense(int T, int H, int E, int k, int I, int norm_topk, int act_dtype, const void *x,
                      const void *w_router, const float *bias, const orc_matrix *w_gate,
                      const orc_matrix *w_up, const orc_matrix *w_down, double *out)
{
    double *logits = (double *)malloc(sizeof(double) * (size_t)T * E);
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)T * k);
    double *w = (double *)malloc(sizeof(double) * (size_t)T * k);
    double *mask = (double *)calloc((size_t)T * E, sizeof(double));
    double *row = (double *)malloc(sizeof(double) * (size_t)H);
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    int rc = (logits && ids && w && mask && row && y) ? 0 : -2;
    if (!rc) rc = orc_router_logits(T, H, E, act_dtype, x, w_router, bias, logits);
    if (!rc) rc = orc_select_topk(T, E, k, norm_topk, logits, ids, w, NULL);
    for (int t = 0; t < T && !rc; ++t)
        for (int j = 0; j < k; ++j) mask[(int64_t)t * E + ids[(int64_t)t * k + j]] = w[(int64_t)t * k + j];
    for (int t = 0; t < T && !rc; ++t) {
        widen_row(act_dtype, x, t, H, row);
        double *o = out + (int64_t)t * H;
        for (int c = 0; c < H; ++c) o[c] = 0.0;
        for (int e = 0; e < E && !rc; ++e) {
            rc = orc_expert_mlp(H, I, row, e, w_gate, w_up, w_down, NULL, y);
            for (int c = 0; c < H && !rc; ++c) o[c] += mask[(int64_t)t * E + e] * y[c];
        }
    }
    free(logits); free(ids); free(w); free(mask); free(row); free(y);
    return rc;
}

/* One weight element as the oracle reads it (exposed so tests can pin the 4-bit decoding). */
double orc_weight_at(const orc_matrix *m, int64_t e, int64_t r, int64_t c)
{
    return weight_at(m, e, r, c);
}

/*
 * Pre-router RMSNorm of the Qwen3 decoder layer, the "layernorm" that the unsloth
 * commit page a1bc5cbd73 (compile_walker paragraph) says Inductor fuses with the
 * residual and router pointwise ops.  The pages give no formula; this is the plain
 * RMSNorm definition:
 *   xn[t,h] = hs[t,h] / sqrt(mean_h' hs[t,h']^2 + eps) * gamma[h]
 * in double, hs and gamma widened exactly from the activation dtype.
 */
int orc_rmsnorm(int T, int H, int act_dtype, const void *hs, const void *gamma, double eps, double *xn)
{
    if (T < 0 || H <= 0 || !xn || (T > 0 && (!hs || !gamma)) || eps < 0) return -1;
    for (int t = 0; t < T; ++t) {
        double ss = 0.0;
        for (int h = 0; h < H; ++h) {
            const double v = act_at(act_dtype, hs, (int64_t)t * H + h);
            ss += v * v;
        }
        const double rms = sqrt(ss / H + eps);
        for (int h = 0; h < H; ++h) {
            const double v = act_at(act_dtype, hs, (int64_t)t * H + h);
            xn[(int64_t)t * H + h] = rms > 0.0 ? v / rms * act_at(act_dtype, gamma, h) : 0.0;
        }
    }
    return 0;
}

/*
 * Rounds doubles to bf16 (8 significant bits, round to nearest, ties to even)
 * directly from double, so no intermediate float rounding can move a tie.
 * Values must lie in the normal bf16 range or be zero.
 */
int orc_round_bf16(int64_t n, const double *v, uint16_t *bits)
{
    if (n < 0 || (n > 0 && (!v || !bits))) return -1;
    for (int64_t i = 0; i < n; ++i) {
        const double d = v[i];
        if (d == 0.0) {
            bits[i] = signbit(d) ? 0x8000u : 0u;
            continue;
        }
        int e = 0;
        const double m = frexp(fabs(d), &e);     /* |d| = m * 2^e, m in [0.5, 1) */
        const double q = ldexp(m, 8);            /* [128, 256): 8 significant bits before the point */
        double r = floor(q);
        const double frac = q - r;
        if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
        const float f = (float)ldexp(r, e - 8);  /* exact: r has at most 9 bits and is a power of 2 when 256 */
        uint32_t u;
        memcpy(&u, &f, sizeof u);
        bits[i] = (uint16_t)((u >> 16) | (d < 0 ? 0x8000u : 0u));
    }
    return 0;
}
