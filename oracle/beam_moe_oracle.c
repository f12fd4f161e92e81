/*
 * Beam routed-MoE forward pass: plain CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the checker for the CUDA library, not part of it:
 * only the test-suite, the package's smoke check and the benchmark's CPU-baseline leg load
 * it. It shares no code, header, table or helper with the CUDA library, and it includes
 * nothing of it. It is written to be read against the pages, not to be fast: every step
 * is the plainest loop, sort or sum that states it, in FP64 where the pages fix no
 * precision.
 *
 * What the method computes, per token (sources: the Beam release pages).
 *   [A] "Reflection releases Beam, a 501B open MoE model with 1M context" (Glonce),
 *       Architecture paragraph: the router scores 256 experts with a sigmoid, splits them
 *       into 8 groups of 32, keeps the 4 best groups, then picks the top 8 experts; there
 *       is no shared expert; expert outputs are combined with normalized router weights and
 *       scaled by 2.5; each expert is a SwiGLU MLP of intermediate size 2,560.
 *   [B] transformers "Beam" model doc, Overview, "Sparse MoE" bullet: a learned per-expert
 *       bias balances load (no auxiliary loss); each token is restricted to the best
 *       topk_group of n_group groups; routing weights are normalized and the MoE output is
 *       scaled by routed_scaling_factor.
 *   [C] same page, paragraph after the bullets: routing and the SwiGLU activation are
 *       computed in FP32; router weights and expert bias are FP32; returned router logits
 *       are FP32.
 *   [D] "Reflection releases Beam, an open 501B AI model built for coding agents"
 *       (unicornapi.net), "How Beam is built": same group sizes as DeepSeek-V3, no shared
 *       expert.
 *
 * Readings where the pages are silent (each is an assumption, stated once here):
 *   R1 group score = sum of the two largest biased scores in the group (the DeepSeek-V3
 *      convention that [A] and [D] name but do not write out);
 *   R2 the bias enters selection only; the weights use the unbiased sigmoid scores;
 *   R3 ties go to the lower group index, then to the lower expert index;
 *   R4 experts of groups that were not kept are excluded from the top-8 outright (not
 *      scored as 0);
 *   R5 the scale 2.5 is folded into the weights (sum of weights = 2.5), which equals
 *      scaling the output in exact arithmetic;
 *   R6 SwiGLU(x) = down( silu(gate x) * (up x) ), silu(z) = z * sigmoid(z); no linear
 *      biases (3 * d * I = 39.3M parameters per expert matches "about 39M" in [A]);
 *   R7 top-k slot order is descending biased score.
 *
 * Precision: the logits are accumulated in FP64 and rounded once to FP32 (the pages fix
 * FP32 router numerics [C]); the sigmoid is evaluated in FP64 and rounded to FP32; the
 * biased score is one FP32 add; group scores are one FP32 add; everything after
 * selection (weights, experts, combine) stays in FP64 with no intermediate rounding.
 * Build with -ffp-contract=off so the FP32 adds are single IEEE operations.
 * Inputs are assumed finite.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int d, I, E, n_group, topk_group, top_k;
    double scale;
} oracle_cfg;

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = -1, ORACLE_MISSING_EXPERT = -2, ORACLE_NO_MEM = -3 };

static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_check_cfg(const oracle_cfg *c)
{
    if (!c || c->d <= 0 || c->I <= 0 || c->E <= 0 || c->n_group <= 0) return ORACLE_BAD_ARG;
    if (c->E % c->n_group) return ORACLE_BAD_ARG;
    if (c->topk_group <= 0 || c->topk_group > c->n_group) return ORACLE_BAD_ARG;
    if (c->top_k <= 0 || c->top_k > c->topk_group * (c->E / c->n_group)) return ORACLE_BAD_ARG;
    return ORACLE_OK;
}

/* Router logits [C]: l[t][e] = sum_j x[t][j] * Wr[e][j], FP64 sum, rounded once to FP32. */
int oracle_router_logits(const oracle_cfg *c, const uint16_t *x, const float *wr, int64_t T, float *logits)
{
    if (oracle_check_cfg(c) || T < 0 || (T && (!x || !wr || !logits))) return ORACLE_BAD_ARG;
    #pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; t++) {
        for (int e = 0; e < c->E; e++) {
            double acc = 0.0;
            for (int j = 0; j < c->d; j++)
                acc += bf16_value(x[t * c->d + j]) * (double)wr[(int64_t)e * c->d + j];
            logits[t * c->E + e] = (float)acc;
        }
    }
    return ORACLE_OK;
}

/* An (expert or group) index with the FP32 score it is ranked by. */
typedef struct { float key; int id; } ranked;

/* Ranking order: higher score first; equal scores -> lower index first (R3). */
static int by_score_then_index(const void *pa, const void *pb)
{
    const ranked *a = (const ranked *)pa, *b = (const ranked *)pb;
    if (a->key > b->key) return -1;
    if (a->key < b->key) return 1;
    return (a->id > b->id) - (a->id < b->id);
}

/*
 * Routing of one token from its FP32 logits [A][B][C], following the steps in order:
 *   1. s_e = sigmoid(l_e), FP64 then rounded to FP32;
 *   2. c_e = s_e + b_e, one FP32 add (bias for selection only, R2);
 *   3. group score gs_g = c(1st) + c(2nd) over the group's experts, one FP32 add (R1);
 *   4. keep the topk_group groups with the largest gs (ties -> lower g);
 *   5. among experts of kept groups only (R4), take the top_k largest c (ties -> lower e),
 *      in descending order (R7);
 *   6. w_k = scale * s_{e_k} / sum_k' s_{e_k'} in FP64 (R5).
 * Optional outputs (NULL to skip): s[E], c[E], gs[n_group], groups[topk_group], w64[top_k].
 */
static void route_one(const oracle_cfg *cf, const float *l, const float *bias, int32_t *idx, float *w,
                      float *s_out, float *c_out, float *gs_out, int32_t *groups_out, double *w64_out,
                      ranked *scratch)
{
    const int E = cf->E, G = cf->n_group, S = E / G;
    float *s = (float *)malloc(sizeof(float) * E);
    float *c = (float *)malloc(sizeof(float) * E);
    float *gs = (float *)malloc(sizeof(float) * G);
    unsigned char *kept = (unsigned char *)calloc(G, 1);

    for (int e = 0; e < E; e++) {
        s[e] = (float)(1.0 / (1.0 + exp(-(double)l[e])));   /* step 1 */
        c[e] = s[e] + bias[e];                                 /* step 2 (FP32 add) */
    }
    for (int g = 0; g < G; g++) {                              /* step 3 */
        for (int j = 0; j < S; j++) { scratch[j].key = c[g * S + j]; scratch[j].id = g * S + j; }
        qsort(scratch, S, sizeof(ranked), by_score_then_index);
        gs[g] = (S >= 2) ? scratch[0].key + scratch[1].key : scratch[0].key;
    }
    for (int g = 0; g < G; g++) { scratch[g].key = gs[g]; scratch[g].id = g; }   /* step 4 */
    qsort(scratch, G, sizeof(ranked), by_score_then_index);
    for (int r = 0; r < cf->topk_group; r++) {
        kept[scratch[r].id] = 1;
        if (groups_out) groups_out[r] = scratch[r].id;
    }
    int n_cand = 0;                                            /* step 5 */
    for (int e = 0; e < E; e++)
        if (kept[e / S]) { scratch[n_cand].key = c[e]; scratch[n_cand].id = e; n_cand++; }
    qsort(scratch, n_cand, sizeof(ranked), by_score_then_index);
    double sum = 0.0;                                          /* step 6 */
    for (int k = 0; k < cf->top_k; k++) { idx[k] = scratch[k].id; sum += (double)s[idx[k]]; }
    for (int k = 0; k < cf->top_k; k++) {
        double wk = cf->scale * (double)s[idx[k]] / sum;
        if (w) w[k] = (float)wk;
        if (w64_out) w64_out[k] = wk;
    }
    if (s_out) memcpy(s_out, s, sizeof(float) * E);
    if (c_out) memcpy(c_out, c, sizeof(float) * E);
    if (gs_out) memcpy(gs_out, gs, sizeof(float) * G);
    free(s); free(c); free(gs); free(kept);
}

/* Routing of T tokens from FP32 logits [T][E]. Debug outputs may be NULL. */
int oracle_route(const oracle_cfg *cf, const float *logits, const float *bias, int64_t T,
                 int32_t *idx, float *w, float *s_out, float *c_out, float *gs_out, int32_t *groups_out,
                 double *w64_out)
{
    if (oracle_check_cfg(cf) || T < 0 || (T && (!logits || !bias || !idx))) return ORACLE_BAD_ARG;
    const int E = cf->E, G = cf->n_group, K = cf->top_k, TG = cf->topk_group;
    #pragma omp parallel
    {
        ranked *scratch = (ranked *)malloc(sizeof(ranked) * (E > G ? E : G));
        #pragma omp for schedule(static)
        for (int64_t t = 0; t < T; t++)
            route_one(cf, logits + t * E, bias, idx + t * K, w ? w + t * K : NULL,
                      s_out ? s_out + t * E : NULL, c_out ? c_out + t * E : NULL,
                      gs_out ? gs_out + t * G : NULL, groups_out ? groups_out + t * TG : NULL,
                      w64_out ? w64_out + t * K : NULL, scratch);
        free(scratch);
    }
    return ORACLE_OK;
}

/*
 * One SwiGLU expert [A][C], R6, all in FP64:
 *   g_i = sum_j x_j Wg[i][j],  u_i = sum_j x_j Wu[i][j]   (i < I)
 *   h_i = g_i * sigmoid(g_i) * u_i
 *   y_j = sum_i h_i Wd[j][i]                               (j < d)
 * Wg, Wu are [I][d] and Wd is [d][I], BF16 bit patterns, row-major.
 */
int oracle_expert(int d, int I, const double *x, const uint16_t *wg, const uint16_t *wu, const uint16_t *wd,
                  double *y)
{
    if (d <= 0 || I <= 0 || !x || !wg || !wu || !wd || !y) return ORACLE_BAD_ARG;
    double *h = (double *)malloc(sizeof(double) * I);
    if (!h) return ORACLE_NO_MEM;
    for (int i = 0; i < I; i++) {
        double g = 0.0, u = 0.0;
        for (int j = 0; j < d; j++) {
            g += x[j] * bf16_value(wg[(int64_t)i * d + j]);
            u += x[j] * bf16_value(wu[(int64_t)i * d + j]);
        }
        h[i] = g / (1.0 + exp(-g)) * u;
    }
    for (int j = 0; j < d; j++) {
        double acc = 0.0;
        for (int i = 0; i < I; i++) acc += h[i] * bf16_value(wd[(int64_t)j * I + i]);
        y[j] = acc;
    }
    free(h);
    return ORACLE_OK;
}

/*
 * The MoE block for a list of tokens: route, run the chosen experts, combine.
 *   out[n] = sum_k w_k * expert_{e_k}(x[tokens[n]])   (FP64, k in slot order)
 * x is [T][d] BF16 bits; tokens (n_tokens entries, each in [0,T)) selects the rows to
 * compute, or is NULL for all T rows in order. logits_in, if not NULL, is [T][E] FP32 and
 * replaces the oracle's own logits (so routing can be checked given another
 * implementation's FP32 logits). idx_in, if not NULL, is [n_tokens][top_k] and replaces
 * the selection (the weights are still computed here from the oracle's sigmoid scores of
 * those experts). wg/wu/wd are arrays of E per-expert pointers; an expert that no token
 * routes to may be NULL. out is [n_tokens][d] FP64; idx_out [n_tokens][top_k] and
 * w_out [n_tokens][top_k] may be NULL.
 */
int oracle_forward(const oracle_cfg *cf, const uint16_t *x, int64_t T, const int64_t *tokens, int64_t n_tokens,
                   const float *logits_in, const float *wr, const float *bias, const int32_t *idx_in,
                   const uint16_t *const *wg, const uint16_t *const *wu, const uint16_t *const *wd,
                   double *out, int32_t *idx_out, float *w_out)
{
    if (oracle_check_cfg(cf) || T < 0 || n_tokens < 0) return ORACLE_BAD_ARG;
    if (!tokens) n_tokens = T;
    if (n_tokens == 0) return ORACLE_OK;
    if (!x || !bias || !out || !wg || !wu || !wd || (!logits_in && !wr)) return ORACLE_BAD_ARG;
    const int d = cf->d, E = cf->E, K = cf->top_k;
    for (int64_t n = 0; n < n_tokens; n++)
        if (tokens && (tokens[n] < 0 || tokens[n] >= T)) return ORACLE_BAD_ARG;

    float *l = (float *)malloc(sizeof(float) * n_tokens * E);
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * n_tokens * K);
    double *w64 = (double *)malloc(sizeof(double) * n_tokens * K);
    double *xd = (double *)malloc(sizeof(double) * n_tokens * d);
    float *s = (float *)malloc(sizeof(float) * n_tokens * E);
    if (!l || !idx || !w64 || !xd || !s) { free(l); free(idx); free(w64); free(xd); free(s); return ORACLE_NO_MEM; }

    int rc = ORACLE_OK;
    for (int64_t n = 0; n < n_tokens; n++) {
        int64_t t = tokens ? tokens[n] : n;
        for (int j = 0; j < d; j++) xd[n * d + j] = bf16_value(x[t * d + j]);
        if (logits_in) memcpy(l + n * E, logits_in + t * E, sizeof(float) * E);
        else oracle_router_logits(cf, x + t * d, wr, 1, l + n * E);
    }
    oracle_route(cf, l, bias, n_tokens, idx, NULL, s, NULL, NULL, NULL, w64);
    if (idx_in) {
        /* Selection given from outside: weights from the oracle's own sigmoid scores. */
        for (int64_t n = 0; n < n_tokens; n++) {
            double sum = 0.0;
            for (int k = 0; k < K; k++) {
                int32_t e = idx_in[n * K + k];
                if (e < 0 || e >= E) rc = ORACLE_BAD_ARG;
                else sum += (double)s[n * E + e];
            }
            for (int k = 0; k < K && rc == ORACLE_OK; k++) {
                idx[n * K + k] = idx_in[n * K + k];
                w64[n * K + k] = cf->scale * (double)s[n * E + idx[n * K + k]] / sum;
            }
        }
    }
    for (int64_t n = 0; n < n_tokens * K && rc == ORACLE_OK; n++)
        if (!wg[idx[n]] || !wu[idx[n]] || !wd[idx[n]]) rc = ORACLE_MISSING_EXPERT;

    if (rc == ORACLE_OK) {
        double *y = (double *)malloc(sizeof(double) * n_tokens * K * d);
        if (!y) rc = ORACLE_NO_MEM;
        else {
            #pragma omp parallel for schedule(dynamic, 1)
            for (int64_t nk = 0; nk < n_tokens * K; nk++) {
                int64_t n = nk / K;
                int e = idx[nk];
                oracle_expert(d, cf->I, xd + n * d, wg[e], wu[e], wd[e], y + nk * d);
            }
            for (int64_t n = 0; n < n_tokens; n++)
                for (int j = 0; j < d; j++) {
                    double acc = 0.0;
                    for (int k = 0; k < K; k++) acc += w64[n * K + k] * y[(n * K + k) * d + j];
                    out[n * d + j] = acc;
                }
            free(y);
        }
    }
    if (rc == ORACLE_OK) {
        if (idx_out) memcpy(idx_out, idx, sizeof(int32_t) * n_tokens * K);
        if (w_out) for (int64_t n = 0; n < n_tokens * K; n++) w_out[n] = (float)w64[n];
    }
    free(l); free(idx); free(w64); free(xd); free(s);
    return rc;
}

/*
 * RMSNorm of one row [E] (HF-doc, "Sandwich norms with depth-scaled residuals" bullet:
 * each block is wrapped in an RMSNorm before and after; the paragraph after the bullets:
 * RMSNorm scaling is computed in FP32). Written out in FP64:
 *   y_j = gamma_j * v_j / sqrt( (1/d) sum_i v_i^2 + eps )
 * Readings (R14): the gain multiplies the normalised vector directly (no "1 + gamma"
 * offset); eps is an argument (the pages give no value).
 * gamma is [d] BF16 bits.
 */
int oracle_rmsnorm(int d, const double *v, const uint16_t *gamma, double eps, double *y)
{
    if (d <= 0 || !v || !gamma || !y || !(eps >= 0.0)) return ORACLE_BAD_ARG;
    double ss = 0.0;
    for (int j = 0; j < d; j++) ss += v[j] * v[j];
    const double r = 1.0 / sqrt(ss / (double)d + eps);
    for (int j = 0; j < d; j++) y[j] = bf16_value(gamma[j]) * v[j] * r;
    return ORACLE_OK;
}

/*
 * Depth-scaled residual update ([A] Glonce, paragraph on the residual connections: the
 * input embedding is step 1; at step k the sublayer output is added with weight 1/sqrt(k)
 * while the existing stream keeps weight sqrt((k-1)/k); HF-doc: after k contributions the
 * stream is their sum divided by sqrt(k)):
 *   out_j = sqrt((k-1)/k) * stream_j + sub_j / sqrt(k),   k >= 2.
 */
int oracle_residual(int d, int k, const double *stream, const double *sub, double *out)
{
    if (d <= 0 || k < 2 || !stream || !sub || !out) return ORACLE_BAD_ARG;
    const double a = sqrt((double)(k - 1) / (double)k), b = 1.0 / sqrt((double)k);
    for (int j = 0; j < d; j++) out[j] = a * stream[j] + b * sub[j];
    return ORACLE_OK;
}

/* BF16 bit pattern nearest to v (round to nearest, ties to even), for finite v in the
 * normal range: the significand is cut to 8 bits by rounding in FP64. */
static uint16_t bf16_round(double v)
{
    if (v == 0.0) return (uint16_t)(signbit(v) ? 0x8000u : 0u);
    int e;
    double m = frexp(v, &e);                   /* v = m * 2^e, 0.5 <= |m| < 1 */
    double r = nearbyint(ldexp(m, 8));         /* 8 significant bits, ties to even */
    float f = (float)ldexp(r, e - 8);          /* exact: 8 bits fit FP32 */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* Rounds n FP64 values to BF16 bit patterns (the MoE block's input is a BF16 hidden state). */
int oracle_round_bf16(int64_t n, const double *v, uint16_t *out)
{
    if (n < 0 || (n && (!v || !out))) return ORACLE_BAD_ARG;
    for (int64_t i = 0; i < n; i++) out[i] = bf16_round(v[i]);
    return ORACLE_OK;
}

/*
 * FP8 E4M3 (the FP8 checkpoint format: [Glonce] Hardware paragraph, the FP8 checkpoint;
 * [HF-doc] quantised checkpoints), decoded from the format's definition: bit 7 sign, bits
 * 6-3 exponent with bias 7, bits 2-0 mantissa; exponent 0 is subnormal (m/8 * 2^-6); the
 * codes 0x7F and 0xFF are NaN (returned as NaN); there are no infinities.
 */
static double e4m3_value(uint8_t q)
{
    const int sign = (q >> 7) & 1, e = (q >> 3) & 15, m = q & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

int oracle_e4m3_decode(int64_t n, const uint8_t *q, double *out)
{
    if (n < 0 || (n && (!q || !out))) return ORACLE_BAD_ARG;
    for (int64_t i = 0; i < n; i++) out[i] = e4m3_value(q[i]);
    return ORACLE_OK;
}

/*
 * One SwiGLU expert with FP8 weights, one FP32 scale per output row (weight-only
 * quantisation; the pages give no recipe, this is the per-row reading): the weights are
 * W[r][c] = scale[r] * e4m3(q[r][c]), and the expert is oracle_expert's, all in FP64:
 *   g_i = sum_j x_j Wg[i][j],  u_i = sum_j x_j Wu[i][j],  h_i = g_i sigmoid(g_i) u_i,
 *   y_j = sum_i h_i Wd[j][i]
 * wg_q, wu_q [I][d] with gs, us [I]; wd_q [d][I] with ds [d].
 */
int oracle_expert_fp8(int d, int I, const double *x, const uint8_t *wg_q, const float *gs, const uint8_t *wu_q,
                      const float *us, const uint8_t *wd_q, const float *ds, double *y)
{
    if (d <= 0 || I <= 0 || !x || !wg_q || !gs || !wu_q || !us || !wd_q || !ds || !y) return ORACLE_BAD_ARG;
    double *h = (double *)malloc(sizeof(double) * I);
    if (!h) return ORACLE_NO_MEM;
    for (int i = 0; i < I; i++) {
        double g = 0.0, u = 0.0;
        for (int j = 0; j < d; j++) {
            g += x[j] * ((double)gs[i] * e4m3_value(wg_q[(int64_t)i * d + j]));
            u += x[j] * ((double)us[i] * e4m3_value(wu_q[(int64_t)i * d + j]));
        }
        h[i] = g * u / (1.0 + exp(-g));
    }
    for (int j = 0; j < d; j++) {
        double acc = 0.0;
        for (int i = 0; i < I; i++) acc += h[i] * ((double)ds[j] * e4m3_value(wd_q[(int64_t)j * I + i]));
        y[j] = acc;
    }
    free(h);
    return ORACLE_OK;
}

/*
 * NVFP4 (the NVFP4 checkpoint: [Glonce] Hardware paragraph, about 280 GB on Blackwell;
 * [Atech] "about 4.5 bits with scales"). The pages give the format's name only; this
 * reading takes the public NVFP4 layout: 4-bit E2M1 codes in blocks of 16 consecutive
 * elements along a row, one E4M3 scale per block, and one FP32 scale per tensor (here: per
 * expert matrix). 4 + 8/16 = 4.5 bits per weight.
 * E2M1 from the format's definition: bit 3 sign, bits 2-1 exponent with bias 1, bit 0
 * mantissa; exponent 0 is subnormal (m * 0.5).
 */
static double e2m1_value(uint8_t c)
{
    const int sign = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    const double v = e == 0 ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, e - 1);
    return sign ? -v : v;
}

/* Values of n E2M1 codes given one per byte (low 4 bits). */
int oracle_e2m1_decode(int64_t n, const uint8_t *c, double *out)
{
    if (n < 0 || (n && (!c || !out))) return ORACLE_BAD_ARG;
    for (int64_t i = 0; i < n; i++) out[i] = e2m1_value(c[i] & 15);
    return ORACLE_OK;
}

/*
 * Element c of an NVFP4 matrix row: codes are packed two per byte, element 2k in the low
 * half of byte k and element 2k+1 in its high half (the reading of the packing); the block
 * scale of element c is the E4M3 code bs[c / 16]:
 *   W[r][c] = t * e4m3(bs[r][c / 16]) * e2m1(code of element c of row r)
 */
static double nvfp4_value(const uint8_t *q_row, const uint8_t *bs_row, double t, int c)
{
    const uint8_t byte = q_row[c / 2];
    const uint8_t code = (c & 1) ? (byte >> 4) : (byte & 15);
    return t * e4m3_value(bs_row[c / 16]) * e2m1_value(code);
}

/*
 * One SwiGLU expert with NVFP4 weights (same form as oracle_expert, all in FP64):
 *   wg_q, wu_q [I][d/2] packed codes with block scales gs, us [I][d/16] and tensor scales
 *   gt, ut; wd_q [d][I/2] with ds [d][I/16] and dt. d and I multiples of 16.
 */
int oracle_expert_nvfp4(int d, int I, const double *x, const uint8_t *wg_q, const uint8_t *gs, double gt,
                        const uint8_t *wu_q, const uint8_t *us, double ut, const uint8_t *wd_q, const uint8_t *ds,
                        double dt, double *y)
{
    if (d <= 0 || I <= 0 || d % 16 || I % 16 || !x || !wg_q || !gs || !wu_q || !us || !wd_q || !ds || !y)
        return ORACLE_BAD_ARG;
    double *h = (double *)malloc(sizeof(double) * I);
    if (!h) return ORACLE_NO_MEM;
    for (int i = 0; i < I; i++) {
        double g = 0.0, u = 0.0;
        const uint8_t *gq = wg_q + (int64_t)i * (d / 2), *gb = gs + (int64_t)i * (d / 16);
        const uint8_t *uq = wu_q + (int64_t)i * (d / 2), *ub = us + (int64_t)i * (d / 16);
        for (int j = 0; j < d; j++) {
            g += x[j] * nvfp4_value(gq, gb, gt, j);
            u += x[j] * nvfp4_value(uq, ub, ut, j);
        }
        h[i] = g * u / (1.0 + exp(-g));
    }
    for (int j = 0; j < d; j++) {
        double acc = 0.0;
        const uint8_t *dq = wd_q + (int64_t)j * (I / 2), *db = ds + (int64_t)j * (I / 16);
        for (int i = 0; i < I; i++) acc += h[i] * nvfp4_value(dq, db, dt, i);
        y[j] = acc;
    }
    free(h);
    return ORACLE_OK;
}
