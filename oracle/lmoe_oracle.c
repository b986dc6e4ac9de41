/*
 * lmoe_oracle.c -- plain, slow, fp64 CPU oracle for the Stable LatentMoE layer
 * forward pass, its backward pass and its Quantile Balancing (QB) histogram /
 * quantile read.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no source, header, table or helper with the CUDA library.
 *
 * Sources (web pages on Kimi K3's architecture):
 *   [DD]  "Kimi-K3-Architecture-Deep-Dive" (jianyuh.github.io)
 *         section 1 "SiTU-GLU", section 2 "Stable LatentMoE", section 3
 *         "Quantile Balancing: A Histogram Trick for 896 Experts".
 *   [IN]  "Inside K3: How Stable Latent MoE and MLA Attention Are Designed"
 *         (besthub.dev), sections "SiTU-GLU", "RMSNorm insertion",
 *         "Quantile Balancing (QB)".
 *   [NW]  "Notes on the MoE and Attention of K3" news write-up (robotbelt.com),
 *         sections "LatentMoE: paying for a bigger pool" and "Keeping the
 *         numbers in range".
 *
 * Every function below is the plain definition, one step at a time, in fp64
 * from the bf16 bit patterns the caller passes (decoded exactly).  Places where
 * the pages are silent carry a "reading:" note; the same readings are listed in
 * the repository's design notes.
 *
 * Build: gcc -O2 -std=c11 -fopenmp -ffp-contract=off -fPIC -shared
 *        (no -ffast-math: the fp32 steps below must be IEEE round-to-nearest).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp64                                                             */
/* ------------------------------------------------------------------------ */

/* Exact decode: a bf16 is the top 16 bits of an IEEE binary32. */
double orc_bf16_to_f64(uint16_t b)
{
    uint32_t bits = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round an fp64 value to the nearest bf16, ties to even, in ONE rounding
 * (no detour through fp32, which could round twice).  bf16 keeps 8
 * significant bits; normal exponents go down to -126, subnormals are spaced
 * 2^-133. */
uint16_t orc_f64_to_bf16(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80);
    int e;
    (void)frexp(a, &e);            /* a = m * 2^e, m in [0.5, 1) */
    int spacing_exp = e - 8;       /* 8 significant bits */
    if (spacing_exp < -133)
        spacing_exp = -133;        /* bf16 subnormal grid */
    double q = ldexp(a, -spacing_exp);       /* exact */
    double qr = nearbyint(q);                /* ties to even (default mode) */
    double v = ldexp(qr, spacing_exp);       /* exact */
    if (v > 3.3895313892515355e38)          /* beyond the largest finite bf16 */
        return (uint16_t)(sign | 0x7F80);
    float f = (float)v;                      /* exact: v has <= 8 bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

static double dot_bf16(const uint16_t *w, const uint16_t *v, int64_t n)
{
    double acc = 0.0;
    for (int64_t i = 0; i < n; ++i)
        acc += orc_bf16_to_f64(w[i]) * orc_bf16_to_f64(v[i]);
    return acc;
}

/* ------------------------------------------------------------------------ */
/* Scalar functions                                                          */
/* ------------------------------------------------------------------------ */

/* Logistic sigmoid 1/(1+e^-x), evaluated without overflow for either sign. */
double orc_sigmoid(double x)
{
    if (x >= 0.0)
        return 1.0 / (1.0 + exp(-x));
    double ex = exp(x);
    return ex / (1.0 + ex);
}

/* [DD] section 1, the SiTU definition: softcap(x; beta) = beta * tanh(x / beta),
 * a smooth bound of x into (-beta, beta). */
double orc_softcap(double x, double beta)
{
    return beta * tanh(x / beta);
}

/* [DD] section 1: SiTU(x; beta) = softcap(x; beta) * sigma(x).  [IN] "SiTU-GLU":
 * the gate is clamped to (-beta, beta) with beta = 4. */
double orc_situ(double x, double beta)
{
    return orc_softcap(x, beta) * orc_sigmoid(x);
}

/* ------------------------------------------------------------------------ */
/* Layer configuration                                                       */
/* ------------------------------------------------------------------------ */

typedef struct {
    int32_t d;            /* hidden size (7168 in K3, [NW] LatentMoE section)   */
    int32_t latent;       /* d/2 latent the routed experts see (3584 in K3)     */
    int32_t n_experts;    /* 2n routed experts (896 in K3)                      */
    int32_t top_k;        /* 2k active per token (16 in K3)                     */
    int32_t inter;        /* routed expert intermediate size                   */
    int32_t n_shared;     /* always-on shared experts (2 in K3)                 */
    int32_t shared_inter; /* intermediate size of each shared expert            */
    double beta1;         /* SiTU cap, 4 ([DD] section 1)                       */
    double beta2;         /* linear-branch softcap, 25 ([DD] section 1)         */
    double rms_eps;       /* reading: 1e-6, inside the square root              */
} orc_config;

/* ------------------------------------------------------------------------ */
/* a1: down-projection d -> d/2, no norm after it                            */
/* ------------------------------------------------------------------------ */

/* [DD] section 2, the LatentMoE diagram: d -> (down) -> d/2 before routing;
 * [DD] section 2 "one RMS Norm before up-projection": the norm after the
 * down-projection was ablated and dropped, so h is the plain linear map.
 * h[t][l] = sum_i W_down[l][i] * x[t][i], in fp64, then rounded once to bf16
 * (reading: the layer's activations are bf16).  w_down is [latent][d]. */
void orc_down_proj(const orc_config *c, int64_t T, const uint16_t *x,
                   const uint16_t *w_down, uint16_t *h_out)
{
    const int64_t d = c->d, L = c->latent;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t l = 0; l < L; ++l)
            h_out[t * L + l] = orc_f64_to_bf16(dot_bf16(w_down + l * d, x + t * d, d));
}

/* Ablation variant: RMSNorm also after the down-projection.  [DD] section 2
 * and [IN] "RMSNorm insertion": the first design put one RMSNorm after the
 * reduction d -> d/2 and one before the expansion; the ablation kept only the
 * second.  This is the first one, for running that variant:
 *   hn[t] = h[t] / sqrt(mean_l h[t][l]^2 + eps)
 * on the bf16 latent h (decoded exactly), in fp64, rounded once to bf16.
 * Reading: un-weighted, with the same eps as the norm before the
 * up-projection. */
void orc_rms_rows(int64_t T, int64_t L, double eps, const uint16_t *h, uint16_t *hn)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double ss = 0.0;
        for (int64_t l = 0; l < L; ++l) {
            const double v = orc_bf16_to_f64(h[t * L + l]);
            ss += v * v;
        }
        const double rms = sqrt(ss / (double)L + eps);
        for (int64_t l = 0; l < L; ++l) {
            const double v = orc_bf16_to_f64(h[t * L + l]);
            hn[t * L + l] = orc_f64_to_bf16(rms > 0.0 ? v / rms : 0.0);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* a2: router scores in the latent                                           */
/* ------------------------------------------------------------------------ */

/* [DD] section 2: routing happens in the d/2 latent, after the down-
 * projection.  Reading: scores are sigma(w_e . h) (the pages only say
 * "router scores"); they lie in (0,1), so the QB map into [0,1] is the
 * identity.  The logit is fp64; the score is stored as fp32.
 * w_router is [n_experts][latent]; s_out is [T][n_experts]. */
void orc_router(const orc_config *c, int64_t T, const uint16_t *h,
                const uint16_t *w_router, float *s_out)
{
    const int64_t L = c->latent, E = c->n_experts;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t e = 0; e < E; ++e)
            s_out[t * E + e] = (float)orc_sigmoid(dot_bf16(w_router + e * L, h + t * L, L));
}

/* ------------------------------------------------------------------------ */
/* a3: biased top-k selection                                                */
/* ------------------------------------------------------------------------ */

typedef struct {
    float u;
    int32_t id;
} scored_id;

/* Larger biased score first; on equal scores the lower expert id first
 * (reading: the pages give no tie rule). */
static int by_score_then_id(const void *pa, const void *pb)
{
    const scored_id *a = (const scored_id *)pa, *b = (const scored_id *)pb;
    if (a->u > b->u) return -1;
    if (a->u < b->u) return 1;
    return (a->id > b->id) - (a->id < b->id);
}

/* [DD] section 3 and [NW] "Keeping the numbers in range": loss-free balancing
 * steers traffic by a per-expert selection bias; the bias changes which
 * experts are chosen, not how their outputs are weighted.
 *   u[t][e] = fp32(s[t][e] + b[e])             (an fp32 add)
 *   idx[t]  = the top_k experts by u, ordered by (u descending, id ascending)
 *   gate[t][j] = s[t][idx[t][j]]                (the unbiased score)
 * Reading: no normalisation of the gates (the RMSNorm after aggregation makes
 * any positive per-token rescaling irrelevant up to eps).
 * margin_out[t] (nullable) = u_(k) - u_(k+1), +inf when top_k == n_experts. */
void orc_topk(const orc_config *c, int64_t T, const float *s, const float *bias,
              int32_t *idx_out, float *gate_out, double *margin_out)
{
    const int64_t E = c->n_experts, K = c->top_k;
#pragma omp parallel
    {
        scored_id *row = (scored_id *)malloc((size_t)E * sizeof(scored_id));
#pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t e = 0; e < E; ++e) {
                float u = s[t * E + e] + bias[e];   /* fp32 + fp32 -> fp32 */
                row[e].u = u;
                row[e].id = (int32_t)e;
            }
            qsort(row, (size_t)E, sizeof(scored_id), by_score_then_id);
            for (int64_t j = 0; j < K; ++j) {
                idx_out[t * K + j] = row[j].id;
                gate_out[t * K + j] = s[t * E + row[j].id];
            }
            if (margin_out)
                margin_out[t] = (K < E) ? (double)row[K - 1].u - (double)row[K].u : INFINITY;
        }
        free(row);
    }
}

/* ------------------------------------------------------------------------ */
/* a4: token permutation (group the T*k assignments by expert)               */
/* ------------------------------------------------------------------------ */

/* Stable counting sort of assignment ids a = t*top_k + j by expert idx[a].
 *   counts[e]   = number of assignments to e
 *   offsets[e]  = exclusive prefix sum of counts (offsets[E] = T*top_k)
 *   perm[p]     = the assignment at permuted row p (experts in id order,
 *                 assignments of one expert in increasing a)
 *   inv[a]      = the permuted row of assignment a (inv[perm[p]] = p). */
void orc_permute(const orc_config *c, int64_t T, const int32_t *idx, int32_t *counts,
                 int32_t *offsets, int32_t *perm, int32_t *inv)
{
    const int64_t E = c->n_experts, N = T * (int64_t)c->top_k;
    for (int64_t e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t a = 0; a < N; ++a)
        counts[idx[a]] += 1;
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int64_t a = 0; a < N; ++a) {
        int32_t e = idx[a];
        int32_t p = offsets[e] + fill[e]++;
        perm[p] = (int32_t)a;
        inv[a] = p;
    }
    free(fill);
}

/* ------------------------------------------------------------------------ */
/* a5 + a6 + a7: routed SiTU-GLU experts, gate-weighted combine, RMSNorm     */
/* ------------------------------------------------------------------------ */

/* One routed expert on one latent row, [DD] section 1:
 *   p1 = W1 h, p2 = W2 h                     (W1, W2: [inter][latent])
 *   act = SiTU(p1; beta1) * softcap(p2; beta2), rounded to bf16
 *         (reading: the expert's intermediate activation is stored in bf16)
 *   o  = W3 act                              (W3: [latent][inter])
 * |SiTU| < beta1 and |softcap| < beta2, so |act| < beta1*beta2 = 100. */
static void expert_row(const orc_config *c, const uint16_t *w1, const uint16_t *w2,
                       const uint16_t *w3, const uint16_t *h, uint16_t *act, double *o)
{
    const int64_t L = c->latent, I = c->inter;
    for (int64_t i = 0; i < I; ++i) {
        double p1 = dot_bf16(w1 + i * L, h, L);
        double p2 = dot_bf16(w2 + i * L, h, L);
        act[i] = orc_f64_to_bf16(orc_situ(p1, c->beta1) * orc_softcap(p2, c->beta2));
    }
    for (int64_t l = 0; l < L; ++l)
        o[l] = dot_bf16(w3 + l * I, act, I);
}

/* Routed branch for every token:
 *   z[t] = sum_j gate[t][j] * E_{idx[t][j]}(h[t])        ([NW]: aggregation)
 *   r[t] = z[t] / sqrt(mean_l z[t][l]^2 + eps)          ([DD] section 2 and
 *          [IN] "RMSNorm insertion": the single norm sits after aggregation and
 *          before the up-projection; reading: no learnable scale, eps = 1e-6)
 * w1[e], w2[e], w3[e] point at expert e's matrices (an expert no token uses may
 * be NULL).  Outputs (each nullable): act_out [T*top_k][inter] bf16 in
 * assignment order, o_out [T*top_k][latent] fp64 gate-weighted expert outputs,
 * z_out [T][latent] fp64, r_out [T][latent] bf16, r64_out [T][latent] fp64. */
void orc_routed(const orc_config *c, int64_t T, const uint16_t *h, const int32_t *idx,
                const float *gate, const uint16_t *const *w1, const uint16_t *const *w2,
                const uint16_t *const *w3, uint16_t *act_out, double *o_out, double *z_out,
                uint16_t *r_out, double *r64_out)
{
    const int64_t L = c->latent, I = c->inter, K = c->top_k;
#pragma omp parallel
    {
        uint16_t *act = (uint16_t *)malloc((size_t)I * sizeof(uint16_t));
        double *o = (double *)malloc((size_t)L * sizeof(double));
        double *z = (double *)malloc((size_t)L * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t l = 0; l < L; ++l)
                z[l] = 0.0;
            for (int64_t j = 0; j < K; ++j) {
                int64_t a = t * K + j;
                int32_t e = idx[a];
                double g = (double)gate[a];
                expert_row(c, w1[e], w2[e], w3[e], h + t * L, act, o);
                for (int64_t l = 0; l < L; ++l)
                    z[l] += g * o[l];
                if (act_out)
                    memcpy(act_out + a * I, act, (size_t)I * sizeof(uint16_t));
                if (o_out)
                    for (int64_t l = 0; l < L; ++l)
                        o_out[a * L + l] = g * o[l];
            }
            double ss = 0.0;
            for (int64_t l = 0; l < L; ++l)
                ss += z[l] * z[l];
            double inv_rms = 1.0 / sqrt(ss / (double)L + c->rms_eps);
            for (int64_t l = 0; l < L; ++l) {
                double r = z[l] * inv_rms;
                if (z_out) z_out[t * L + l] = z[l];
                if (r_out) r_out[t * L + l] = orc_f64_to_bf16(r);
                if (r64_out) r64_out[t * L + l] = r;
            }
        }
        free(act);
        free(o);
        free(z);
    }
}

/* The aggregation of the routed experts from given activations ([DD] section
 * 2 and [NW] "Keeping the numbers in range": the routed outputs are summed,
 * gate-weighted, before the single norm):
 *   z[t] = sum_j gate[t][j] * W3[idx[t][j]] act[t*top_k + j]
 * act: [T*top_k][inter] bf16 in assignment order (e.g. another
 * implementation's activations, to check its aggregation alone); z_out
 * [T][latent] fp64.  The same products and sums, in the same order, as the
 * aggregation inside orc_routed. */
void orc_expert_aggregate(const orc_config *c, int64_t T, const uint16_t *act, const int32_t *idx,
                          const float *gate, const uint16_t *const *w3, double *z_out)
{
    const int64_t L = c->latent, I = c->inter, K = c->top_k;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        double *z = z_out + t * L;
        for (int64_t l = 0; l < L; ++l)
            z[l] = 0.0;
        for (int64_t j = 0; j < K; ++j) {
            const int64_t a = t * K + j;
            const double g = (double)gate[a];
            const uint16_t *w = w3[idx[a]];
            for (int64_t l = 0; l < L; ++l)
                z[l] += g * dot_bf16(w + l * I, act + a * I, I);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* FP8 variant of the routed experts (e4m3 weights and activations)          */
/* ------------------------------------------------------------------------ */

/* [NW] "Keeping the numbers in range": SiTU-GLU bounds the expert activation
 * (|act| < beta1*beta2 = 100), which is what makes low-precision experts
 * practical.  The pages give no FP8 recipe; the reading implemented here:
 *   - e4m3 (OCP FP8: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 *     bits; no infinities; largest finite 448 = 1.75 * 2^8; smallest normal
 *     2^-6; subnormals k * 2^-9), round to nearest even, saturating at +-448;
 *   - every weight row (one output channel of W1, W2 or W3 of one expert) and
 *     every token's latent row gets a power-of-two scale 2^e, e the smallest
 *     integer with max|row| <= 448 * 2^e (0 for an all-zero row); a code is
 *     e4m3(v * 2^-e) -- the scaling is exact, so only the e4m3 rounding acts;
 *   - the expert activation uses the fixed scale 2^-2: act8 = e4m3(4 * act),
 *     which never saturates because |4 * act| < 400 <= 448;
 *   - dot products of the decoded values in fp64, then the two power-of-two
 *     scales. */

double orc_e4m3_to_f64(uint8_t c)
{
    const int sign = c >> 7, ex = (c >> 3) & 15, m = c & 7;
    if (ex == 15 && m == 7)
        return NAN;
    double v = (ex == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, ex - 7);
    return sign ? -v : v;
}

uint8_t orc_f64_to_e4m3(double x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs(x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);          /* saturate (also +-inf) */
    if (a < ldexp(1.0, -6)) {                   /* subnormal grid k * 2^-9 */
        double k = nearbyint(ldexp(a, 9));      /* ties to even */
        return (uint8_t)(sign | (uint8_t)k);    /* k = 8 is the smallest normal */
    }
    int e;
    (void)frexp(a, &e);                         /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;                                     /* a = (1 + m) * 2^e */
    double q = nearbyint(ldexp(a, 3 - e));      /* 8..16, ties to even */
    if (q == 16.0) {
        q = 8.0;
        e += 1;
    }
    if (e > 8 || (e == 8 && q > 14.0))          /* past 448 after rounding */
        return (uint8_t)(sign | 0x7E);
    return (uint8_t)(sign | (uint8_t)((e + 7) << 3) | (uint8_t)(q - 8.0));
}

/* Smallest integer e with amax <= 448 * 2^e (amax >= 0); 0 for amax = 0.
 * With amax = f * 2^x, f in [0.5, 1), and 448 = 0.875 * 2^9. */
int32_t orc_fp8_exp_for(double amax)
{
    if (!(amax > 0.0))
        return 0;
    int x;
    double f = frexp(amax, &x);
    return (f <= 0.875) ? x - 9 : x - 8;
}

/* codes[r][k] = e4m3(src[r][k] * 2^-exps[r]) for the R rows of K bf16 values. */
void orc_fp8_quantize_rows(const uint16_t *src, int64_t R, int64_t K, uint8_t *codes, int8_t *exps)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        double amax = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double v = fabs(orc_bf16_to_f64(src[r * K + k]));
            if (v > amax) amax = v;
        }
        const int32_t e = orc_fp8_exp_for(amax);
        exps[r] = (int8_t)e;
        for (int64_t k = 0; k < K; ++k)
            codes[r * K + k] = orc_f64_to_e4m3(ldexp(orc_bf16_to_f64(src[r * K + k]), -e));
    }
}

static double dot_e4m3(const uint8_t *a, const uint8_t *b, int64_t n)
{
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i)
        s += orc_e4m3_to_f64(a[i]) * orc_e4m3_to_f64(b[i]);
    return s;
}

/* The routed branch with e4m3 experts (same structure as orc_routed):
 *   h8, he  = quantised latent row of the token
 *   p1[f]   = (h8 . w1q[f]) * 2^(he + w1e[f]),  p2 likewise with W2
 *   act8[f] = e4m3(4 * SiTU(p1[f]; beta1) * softcap(p2[f]; beta2))
 *   o[l]    = (act8 . w3q[l]) * 2^(w3e[l] - 2)
 *   z, r    as in orc_routed.
 * Per expert e: w1q[e], w2q[e] [inter][latent] codes with w1e[e], w2e[e]
 * [inter] exponents; w3q[e] [latent][inter] with w3e[e] [latent].  Outputs
 * (nullable): act8_out [T*top_k][inter] codes in assignment order, o_out
 * [T*top_k][latent] fp64 (gate-weighted), z_out, r_out (bf16), r64_out. */
void orc_routed_fp8(const orc_config *c, int64_t T, const uint16_t *h, const int32_t *idx,
                    const float *gate, const uint8_t *const *w1q, const int8_t *const *w1e,
                    const uint8_t *const *w2q, const int8_t *const *w2e, const uint8_t *const *w3q,
                    const int8_t *const *w3e, uint8_t *act8_out, double *o_out, double *z_out,
                    uint16_t *r_out, double *r64_out)
{
    const int64_t L = c->latent, I = c->inter, K = c->top_k;
#pragma omp parallel
    {
        uint8_t *h8 = (uint8_t *)malloc((size_t)L);
        uint8_t *act8 = (uint8_t *)malloc((size_t)I);
        double *z = (double *)malloc((size_t)L * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
            int8_t he;
            orc_fp8_quantize_rows(h + t * L, 1, L, h8, &he);
            for (int64_t l = 0; l < L; ++l)
                z[l] = 0.0;
            for (int64_t j = 0; j < K; ++j) {
                const int64_t a = t * K + j;
                const int32_t e = idx[a];
                const double g = (double)gate[a];
                for (int64_t f = 0; f < I; ++f) {
                    double p1 = ldexp(dot_e4m3(h8, w1q[e] + f * L, L), he + w1e[e][f]);
                    double p2 = ldexp(dot_e4m3(h8, w2q[e] + f * L, L), he + w2e[e][f]);
                    act8[f] = orc_f64_to_e4m3(4.0 * orc_situ(p1, c->beta1) * orc_softcap(p2, c->beta2));
                }
                if (act8_out)
                    memcpy(act8_out + a * I, act8, (size_t)I);
                for (int64_t l = 0; l < L; ++l) {
                    const double o = ldexp(dot_e4m3(act8, w3q[e] + l * I, I), w3e[e][l] - 2);
                    z[l] += g * o;
                    if (o_out)
                        o_out[a * L + l] = g * o;
                }
            }
            double ss = 0.0;
            for (int64_t l = 0; l < L; ++l)
                ss += z[l] * z[l];
            const double inv_rms = 1.0 / sqrt(ss / (double)L + c->rms_eps);
            for (int64_t l = 0; l < L; ++l) {
                const double r = z[l] * inv_rms;
                if (z_out) z_out[t * L + l] = z[l];
                if (r_out) r_out[t * L + l] = orc_f64_to_bf16(r);
                if (r64_out) r64_out[t * L + l] = r;
            }
        }
        free(h8);
        free(act8);
        free(z);
    }
}

/* ------------------------------------------------------------------------ */
/* a8: shared experts and the up-projection                                  */
/* ------------------------------------------------------------------------ */

/* [NW] "LatentMoE": two shared experts always participate.  Reading: each is
 * a SiTU-GLU expert d -> shared_inter -> d acting on x itself, added after the
 * up-projection.  ws1, ws2 are [n_shared*shared_inter][d] (expert s owns rows
 * s*shared_inter ...); the activation is rounded to bf16:
 *   as[t][s*Is + i] = bf16(SiTU(ws1[s*Is+i] . x[t]; beta1) * softcap(ws2[s*Is+i] . x[t]; beta2)) */
void orc_shared_act(const orc_config *c, int64_t T, const uint16_t *x, const uint16_t *ws1,
                    const uint16_t *ws2, uint16_t *as_out)
{
    const int64_t d = c->d, S = (int64_t)c->n_shared * c->shared_inter;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t i = 0; i < S; ++i) {
            double p1 = dot_bf16(ws1 + i * d, x + t * d, d);
            double p2 = dot_bf16(ws2 + i * d, x + t * d, d);
            as_out[t * S + i] = orc_f64_to_bf16(orc_situ(p1, c->beta1) * orc_softcap(p2, c->beta2));
        }
}

/* [DD] section 2: d/2 -> (up) -> d after the norm; plus the shared experts'
 * W3 (ws3 is [d][n_shared*shared_inter], expert s owns columns s*Is ...):
 *   y[t][m] = sum_l W_up[m][l] r[t][l] + sum_s sum_i ws3[m][s*Is+i] as[t][s*Is+i]
 * w_up is [d][latent].  r is the bf16 normalised latent.  No residual add
 * (the residual stream is outside the layer).  y is fp64. */
void orc_up_shared(const orc_config *c, int64_t T, const uint16_t *r, const uint16_t *as,
                   const uint16_t *w_up, const uint16_t *ws3, double *y_out)
{
    const int64_t d = c->d, L = c->latent, Is = c->shared_inter, ns = c->n_shared;
    const int64_t S = ns * Is;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t m = 0; m < d; ++m) {
            double acc = dot_bf16(w_up + m * L, r + t * L, L);
            for (int64_t s = 0; s < ns; ++s)
                for (int64_t i = 0; i < Is; ++i)
                    acc += orc_bf16_to_f64(ws3[m * S + s * Is + i]) *
                           orc_bf16_to_f64(as[t * S + s * Is + i]);
            y_out[t * d + m] = acc;
        }
}

/* ------------------------------------------------------------------------ */
/* a9: QB histogram                                                          */
/* ------------------------------------------------------------------------ */

/* [DD] section 3, steps 1-2 and [IN] "Quantile Balancing (QB)": map the
 * scores into [0,1] (the identity for sigmoid scores) and keep a B-bin
 * frequency histogram per expert over all scores, biased or not chosen.
 *   bin(s) = min(B-1, floor(fp32(s * B)))   -- fp32 multiply, then floor
 *   hist[e][bin(s[t][e])] += 1   for every token t
 * s has row stride ld (elements).  accumulate = 0 clears hist first; 1 adds
 * to it (histograms are additive, [DD] section 3 step 3).  Reading: scores
 * below 0 go to bin 0 (they cannot occur for sigmoid outputs). */
void orc_qb_histogram(const float *s, int64_t T, int32_t E, int64_t ld, int32_t B,
                      uint32_t *hist, int accumulate)
{
    if (!accumulate)
        memset(hist, 0, (size_t)E * (size_t)B * sizeof(uint32_t));
    const float fB = (float)B;
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < E; ++e)
        for (int64_t t = 0; t < T; ++t) {
            float v = s[t * ld + e] * fB;   /* one fp32 rounding */
            float f = floorf(v);
            int64_t bin = (f < 0.0f) ? 0 : (int64_t)f;
            if (bin > B - 1)
                bin = B - 1;
            hist[e * (int64_t)B + bin] += 1u;
        }
}

/* ------------------------------------------------------------------------ */
/* a10: QB quantile read -> per-expert bias                                  */
/* ------------------------------------------------------------------------ */

/* [DD] section 3 (QB replaces the fixed-step bias update; zero extra
 * hyper-parameters), [IN] "Quantile Balancing (QB)" (read the quantile from
 * the histogram) and [NW] "Keeping the numbers in range" (estimate where
 * each expert's threshold must sit to receive its target share).
 * Reading, per expert e:
 *   N      = sum_j hist[e][j]
 *   r      = clamp(ceil(level * N), 1, N)            (rank of the quantile)
 *   C_j    = hist[e][0] + ... + hist[e][j]
 *   j*     = min { j : C_j >= r }
 *   q[e]   = (j* + (r - C_{j*-1}) / hist[e][j*]) / B  (linear inside the bin)
 *   b[e]   = -q[e]
 * level = 1 - top_k/n_experts.  With b = -q every expert clears a common
 * threshold of 0 on a top_k/n_experts share of tokens.  An empty row
 * (N = 0) gives q = 0, b = 0.  q_out is nullable. */
void orc_qb_quantile_bias(const uint32_t *hist, int32_t E, int32_t B, double level,
                          float *q_out, float *b_out)
{
    for (int64_t e = 0; e < E; ++e) {
        const uint32_t *row = hist + e * (int64_t)B;
        uint64_t n = 0;
        for (int64_t j = 0; j < B; ++j)
            n += row[j];
        double q = 0.0;
        if (n > 0) {
            double rr = ceil(level * (double)n);
            if (rr < 1.0) rr = 1.0;
            if (rr > (double)n) rr = (double)n;
            uint64_t r = (uint64_t)rr;
            uint64_t below = 0;   /* C_{j-1} */
            for (int64_t j = 0; j < B; ++j) {
                if (below + row[j] >= r) {
                    q = ((double)j + (double)(r - below) / (double)row[j]) / (double)B;
                    break;
                }
                below += row[j];
            }
        }
        if (q_out) q_out[e] = (float)q;
        b_out[e] = (float)(-q);
    }
}

/* ------------------------------------------------------------------------ */
/* The fixed-step bias update QB replaces (closed-loop comparison)           */
/* ------------------------------------------------------------------------ */

/* [NW] "Keeping the numbers in range" and [DD] section 3: K2's loss-free
 * balancing changed each expert's selection bias by a constant amount per
 * update, in the direction of its load error only (the page likens it to
 * SignSGD).  Reading (the pages give no formula):
 *   mean   = (counts[0] + ... + counts[E-1]) / E
 *   b[e]  += gamma * sign(mean - counts[e]),   sign(0) = 0
 * An under-loaded expert's bias rises, an over-loaded one's falls.  The
 * comparison is done exactly in integers (counts[e] * E against the total);
 * the add is one fp32 addition. */
void orc_sign_update(const int32_t *counts, int32_t E, float gamma, float *bias)
{
    int64_t total = 0;
    for (int64_t e = 0; e < E; ++e)
        total += counts[e];
    for (int64_t e = 0; e < E; ++e) {
        const int64_t scaled = (int64_t)counts[e] * (int64_t)E;
        if (scaled < total)
            bias[e] = bias[e] + gamma;
        else if (scaled > total)
            bias[e] = bias[e] - gamma;
    }
}

/* ------------------------------------------------------------------------ */
/* Backward pass of the layer                                                */
/* ------------------------------------------------------------------------ */

/* [DD] section 1: the tanh softcap is continuous and differentiable everywhere:
 *   d/dx softcap(x; beta) = 1 - tanh(x / beta)^2
 *   d/dx SiTU(x; beta)    = softcap'(x) sigma(x) + softcap(x) sigma(x) (1 - sigma(x)) */
double orc_softcap_grad(double x, double beta)
{
    double t = tanh(x / beta);
    return 1.0 - t * t;
}

double orc_situ_grad(double x, double beta)
{
    double s = orc_sigmoid(x);
    return orc_softcap_grad(x, beta) * s + orc_softcap(x, beta) * s * (1.0 - s);
}

static double dot_bf16_f64(const uint16_t *w, const double *v, int64_t n)
{
    double acc = 0.0;
    for (int64_t i = 0; i < n; ++i)
        acc += orc_bf16_to_f64(w[i]) * v[i];
    return acc;
}

static double keep(double v, int round_mode)
{
    return round_mode ? orc_bf16_to_f64(orc_f64_to_bf16(v)) : v;
}

/* Gradient of the layer y(x) (the forward above) for an upstream gradient dy,
 * with the forward's routing idx held fixed: the top-k choice has no
 * gradient; the router's gradient flows through the gates
 * g_j = sigma(w_router[e_j] . h).  The selection bias never enters y.
 *
 * round_mode 1: the forward's roundings (h, act, r and the shared activation
 * in bf16, the gates in fp32) are applied to the values the gradient is taken
 * at, and each rounding passes the gradient through unchanged.  round_mode 0:
 * no rounding anywhere -- the gradient of the smooth function, which
 * finite differences can check.
 *
 * Per token (tokens are independent):
 *   dr  = W_up^T dy                 das  = Ws3^T dy
 *   dps1 = das SiTU'(ps1) softcap(ps2)   dps2 = das SiTU(ps1) softcap'(ps2)
 *   RMSNorm r = z / sqrt(ms + eps), ms = mean(z^2):
 *   dz  = dr / sqrt(ms + eps) - z (dr . z) / (L (ms + eps)^(3/2))
 *   per chosen expert j (e = idx, o_j = W3[e] act_j, the gate not applied):
 *     dg_j = o_j . dz      do_j = g_j dz      dact_j = W3[e]^T do_j
 *     dp1_j = dact_j SiTU'(p1_j) softcap(p2_j)
 *     dp2_j = dact_j SiTU(p1_j) softcap'(p2_j)
 *     dlogit_j = dg_j sigma'(logit_j),  sigma'(x) = sigma(x) sigma(-x)
 *     dh += W1[e]^T dp1_j + W2[e]^T dp2_j + w_router[e] dlogit_j
 *   dx  = W_down^T dh + Ws1^T dps1 + Ws2^T dps2
 * Weights (sums over tokens in ascending order, over an expert's assignments
 * in ascending assignment order):
 *   dW_up = sum dy r^T  ([DD] section 2, effect 6: the gradient of the
 *           projection after the norm is the outer product with the
 *           normalised latent)
 *   dWs3 = sum dy as^T, dWs1 = sum dps1 x^T, dWs2 = sum dps2 x^T,
 *   dW_down = sum dh x^T, dW_router[e] = sum dlogit h^T,
 *   dW3[e] = sum do act^T, dW1[e] = sum dp1 h^T, dW2[e] = sum dp2 h^T.
 * Layouts as the weights: dw_down [L][d], dw_router [E][L], dw1/dw2 [E][I][L],
 * dw3 [E][L][I], dws1/dws2 [S][d], dws3 [d][S], dw_up [d][L]; dx [T][d].
 * Every output is nullable (a NULL weight gradient skips its sum).  w1, w2,
 * w3 are per-expert pointers as in orc_routed.
 * norm_after_down (the ablation variant): the latent the router and the
 * experts see is h = h_raw / sqrt(mean(h_raw^2) + eps) of the down-
 * projection's h_raw, so the gradient dh reaching it goes through the same
 * RMSNorm backward as dz above before the down-projection:
 *   dh_raw = dh / sqrt(ms + eps) - h_raw (dh . h_raw) / (L (ms + eps)^(3/2)),
 * and dx and dW_down use dh_raw. */
void orc_backward(const orc_config *c, int64_t T, const uint16_t *x, const int32_t *idx,
                  const uint16_t *dy, const uint16_t *w_down, const uint16_t *w_router,
                  const uint16_t *const *w1, const uint16_t *const *w2, const uint16_t *const *w3,
                  const uint16_t *ws1, const uint16_t *ws2, const uint16_t *ws3,
                  const uint16_t *w_up, int round_mode, int norm_after_down, double *dx,
                  double *dw_down, double *dw_router, double *dw1, double *dw2, double *dw3,
                  double *dws1, double *dws2, double *dws3, double *dw_up)
{
    const int64_t d = c->d, L = c->latent, E = c->n_experts, K = c->top_k, I = c->inter;
    const int64_t S = (int64_t)c->n_shared * c->shared_inter;
    const int64_t n = T * K;
    const double b1 = c->beta1, b2 = c->beta2;
    /* values kept per token / per assignment for the weight sums */
    double *hv = (double *)malloc((size_t)(T * L) * sizeof(double));
    double *rv = (double *)malloc((size_t)(T * L) * sizeof(double));
    double *asv = (double *)malloc((size_t)(T * S) * sizeof(double));
    double *dps1v = (double *)malloc((size_t)(T * S) * sizeof(double));
    double *dps2v = (double *)malloc((size_t)(T * S) * sizeof(double));
    double *dhv = (double *)malloc((size_t)(T * L) * sizeof(double));
    double *dlgv = (double *)malloc((size_t)n * sizeof(double));
    double *dov = (double *)malloc((size_t)(n * L) * sizeof(double));
    double *actv = (double *)malloc((size_t)(n * I) * sizeof(double));
    double *dp1v = (double *)malloc((size_t)(n * I) * sizeof(double));
    double *dp2v = (double *)malloc((size_t)(n * I) * sizeof(double));

#pragma omp parallel
    {
        double *xd = (double *)malloc((size_t)d * sizeof(double));
        double *dyd = (double *)malloc((size_t)d * sizeof(double));
        double *hraw = (double *)malloc((size_t)L * sizeof(double));
        double *ps1 = (double *)malloc((size_t)S * sizeof(double));
        double *ps2 = (double *)malloc((size_t)S * sizeof(double));
        double *p1 = (double *)malloc((size_t)(K * I) * sizeof(double));
        double *p2 = (double *)malloc((size_t)(K * I) * sizeof(double));
        double *o = (double *)malloc((size_t)(K * L) * sizeof(double));
        double *g = (double *)malloc((size_t)K * sizeof(double));
        double *dsig = (double *)malloc((size_t)K * sizeof(double));
        double *z = (double *)malloc((size_t)L * sizeof(double));
        double *dr = (double *)malloc((size_t)L * sizeof(double));
        double *dz = (double *)malloc((size_t)L * sizeof(double));
        double *das = (double *)malloc((size_t)S * sizeof(double));
        double *dact = (double *)malloc((size_t)I * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
            double *h = hv + t * L, *dh = dhv + t * L;
            for (int64_t q = 0; q < d; ++q) {
                xd[q] = orc_bf16_to_f64(x[t * d + q]);
                dyd[q] = orc_bf16_to_f64(dy[t * d + q]);
            }
            /* forward values */
            for (int64_t l = 0; l < L; ++l)
                hraw[l] = keep(dot_bf16_f64(w_down + l * d, xd, d), round_mode);
            double den_h = 1.0, inv_h = 1.0;
            if (norm_after_down) {
                double msh = 0.0;
                for (int64_t l = 0; l < L; ++l)
                    msh += hraw[l] * hraw[l];
                den_h = msh / (double)L + c->rms_eps;
                inv_h = 1.0 / sqrt(den_h);
            }
            for (int64_t l = 0; l < L; ++l)
                h[l] = norm_after_down ? keep(hraw[l] * inv_h, round_mode) : hraw[l];
            for (int64_t i = 0; i < S; ++i) {
                ps1[i] = dot_bf16_f64(ws1 + i * d, xd, d);
                ps2[i] = dot_bf16_f64(ws2 + i * d, xd, d);
                asv[t * S + i] = keep(orc_situ(ps1[i], b1) * orc_softcap(ps2[i], b2), round_mode);
            }
            for (int64_t l = 0; l < L; ++l)
                z[l] = 0.0;
            for (int64_t j = 0; j < K; ++j) {
                const int64_t a = t * K + j;
                const int32_t e = idx[a];
                const double logit = dot_bf16_f64(w_router + (int64_t)e * L, h, L);
                const double sig = orc_sigmoid(logit);
                g[j] = round_mode ? (double)(float)sig : sig;
                /* sigma'(x) = sigma(x) sigma(-x): no cancellation in 1 - sigma
                 * where sigma(x) rounds to 1 */
                dsig[j] = sig * orc_sigmoid(-logit);
                for (int64_t i = 0; i < I; ++i) {
                    p1[j * I + i] = dot_bf16_f64(w1[e] + i * L, h, L);
                    p2[j * I + i] = dot_bf16_f64(w2[e] + i * L, h, L);
                    actv[a * I + i] = keep(orc_situ(p1[j * I + i], b1) * orc_softcap(p2[j * I + i], b2),
                                           round_mode);
                }
                for (int64_t l = 0; l < L; ++l) {
                    o[j * L + l] = dot_bf16_f64(w3[e] + l * I, actv + a * I, I);
                    z[l] += g[j] * o[j * L + l];
                }
            }
            double ms = 0.0;
            for (int64_t l = 0; l < L; ++l)
                ms += z[l] * z[l];
            const double den = ms / (double)L + c->rms_eps;
            const double inv = 1.0 / sqrt(den);
            for (int64_t l = 0; l < L; ++l)
                rv[t * L + l] = keep(z[l] * inv, round_mode);
            /* up-projection and shared experts */
            for (int64_t l = 0; l < L; ++l)
                dr[l] = 0.0;
            for (int64_t i = 0; i < S; ++i)
                das[i] = 0.0;
            for (int64_t m = 0; m < d; ++m) {
                for (int64_t l = 0; l < L; ++l)
                    dr[l] += orc_bf16_to_f64(w_up[m * L + l]) * dyd[m];
                for (int64_t i = 0; i < S; ++i)
                    das[i] += orc_bf16_to_f64(ws3[m * S + i]) * dyd[m];
            }
            for (int64_t i = 0; i < S; ++i) {
                dps1v[t * S + i] = das[i] * orc_situ_grad(ps1[i], b1) * orc_softcap(ps2[i], b2);
                dps2v[t * S + i] = das[i] * orc_situ(ps1[i], b1) * orc_softcap_grad(ps2[i], b2);
            }
            /* RMSNorm */
            double drz = 0.0;
            for (int64_t l = 0; l < L; ++l)
                drz += dr[l] * z[l];
            for (int64_t l = 0; l < L; ++l)
                dz[l] = dr[l] * inv - z[l] * drz * inv / ((double)L * den);
            /* routed experts, gates and router */
            for (int64_t l = 0; l < L; ++l)
                dh[l] = 0.0;
            for (int64_t j = 0; j < K; ++j) {
                const int64_t a = t * K + j;
                const int32_t e = idx[a];
                double dg = 0.0;
                for (int64_t l = 0; l < L; ++l) {
                    dg += o[j * L + l] * dz[l];
                    dov[a * L + l] = g[j] * dz[l];
                }
                for (int64_t i = 0; i < I; ++i)
                    dact[i] = 0.0;
                for (int64_t l = 0; l < L; ++l) {
                    const uint16_t *w3row = w3[e] + l * I;
                    for (int64_t i = 0; i < I; ++i)
                        dact[i] += orc_bf16_to_f64(w3row[i]) * dov[a * L + l];
                }
                for (int64_t i = 0; i < I; ++i) {
                    const double x1 = p1[j * I + i], x2 = p2[j * I + i];
                    const double d1 = dact[i] * orc_situ_grad(x1, b1) * orc_softcap(x2, b2);
                    const double d2 = dact[i] * orc_situ(x1, b1) * orc_softcap_grad(x2, b2);
                    dp1v[a * I + i] = d1;
                    dp2v[a * I + i] = d2;
                    const uint16_t *r1 = w1[e] + i * L, *r2 = w2[e] + i * L;
                    for (int64_t l = 0; l < L; ++l)
                        dh[l] += orc_bf16_to_f64(r1[l]) * d1 + orc_bf16_to_f64(r2[l]) * d2;
                }
                dlgv[a] = dg * dsig[j];
                for (int64_t l = 0; l < L; ++l)
                    dh[l] += orc_bf16_to_f64(w_router[(int64_t)e * L + l]) * dlgv[a];
            }
            /* the variant's RMSNorm after the down-projection */
            if (norm_after_down) {
                double dhh = 0.0;
                for (int64_t l = 0; l < L; ++l)
                    dhh += dh[l] * hraw[l];
                for (int64_t l = 0; l < L; ++l)
                    dh[l] = dh[l] * inv_h - hraw[l] * dhh * inv_h / ((double)L * den_h);
            }
            /* down-projection and the shared experts' input side */
            if (dx) {
                double *dxt = dx + t * d;
                for (int64_t q = 0; q < d; ++q)
                    dxt[q] = 0.0;
                for (int64_t l = 0; l < L; ++l)
                    for (int64_t q = 0; q < d; ++q)
                        dxt[q] += orc_bf16_to_f64(w_down[l * d + q]) * dh[l];
                for (int64_t i = 0; i < S; ++i)
                    for (int64_t q = 0; q < d; ++q)
                        dxt[q] += orc_bf16_to_f64(ws1[i * d + q]) * dps1v[t * S + i] +
                                  orc_bf16_to_f64(ws2[i * d + q]) * dps2v[t * S + i];
            }
        }
        free(xd); free(dyd); free(hraw); free(ps1); free(ps2); free(p1); free(p2); free(o); free(g);
        free(dsig); free(z); free(dr); free(dz); free(das); free(dact);
    }

    /* weight gradients: one output row per iteration, tokens in order */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < d; ++m) {
        if (dw_up)
            for (int64_t l = 0; l < L; ++l)
                dw_up[m * L + l] = 0.0;
        if (dws3)
            for (int64_t i = 0; i < S; ++i)
                dws3[m * S + i] = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            const double gm = orc_bf16_to_f64(dy[t * d + m]);
            if (dw_up)
                for (int64_t l = 0; l < L; ++l)
                    dw_up[m * L + l] += gm * rv[t * L + l];
            if (dws3)
                for (int64_t i = 0; i < S; ++i)
                    dws3[m * S + i] += gm * asv[t * S + i];
        }
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < S; ++i) {
        for (int64_t q = 0; q < d; ++q) {
            if (dws1) dws1[i * d + q] = 0.0;
            if (dws2) dws2[i * d + q] = 0.0;
        }
        for (int64_t t = 0; t < T; ++t)
            for (int64_t q = 0; q < d; ++q) {
                const double xv = orc_bf16_to_f64(x[t * d + q]);
                if (dws1) dws1[i * d + q] += dps1v[t * S + i] * xv;
                if (dws2) dws2[i * d + q] += dps2v[t * S + i] * xv;
            }
    }
    if (dw_down) {
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t l = 0; l < L; ++l) {
            for (int64_t q = 0; q < d; ++q)
                dw_down[l * d + q] = 0.0;
            for (int64_t t = 0; t < T; ++t)
                for (int64_t q = 0; q < d; ++q)
                    dw_down[l * d + q] += dhv[t * L + l] * orc_bf16_to_f64(x[t * d + q]);
        }
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t e = 0; e < E; ++e) {
        if (dw_router)
            for (int64_t l = 0; l < L; ++l)
                dw_router[e * L + l] = 0.0;
        if (dw3)
            for (int64_t q = 0; q < L * I; ++q)
                dw3[e * L * I + q] = 0.0;
        for (int64_t q = 0; q < I * L; ++q) {
            if (dw1) dw1[e * I * L + q] = 0.0;
            if (dw2) dw2[e * I * L + q] = 0.0;
        }
        for (int64_t a = 0; a < n; ++a) {
            if (idx[a] != e)
                continue;
            const double *h = hv + (a / K) * L;
            if (dw_router)
                for (int64_t l = 0; l < L; ++l)
                    dw_router[e * L + l] += dlgv[a] * h[l];
            if (dw3)
                for (int64_t l = 0; l < L; ++l)
                    for (int64_t i = 0; i < I; ++i)
                        dw3[(e * L + l) * I + i] += dov[a * L + l] * actv[a * I + i];
            for (int64_t i = 0; i < I; ++i)
                for (int64_t l = 0; l < L; ++l) {
                    if (dw1) dw1[(e * I + i) * L + l] += dp1v[a * I + i] * h[l];
                    if (dw2) dw2[(e * I + i) * L + l] += dp2v[a * I + i] * h[l];
                }
        }
    }
    free(hv); free(rv); free(asv); free(dps1v); free(dps2v); free(dhv); free(dlgv); free(dov);
    free(actv); free(dp1v); free(dp2v);
}

/* Number of OpenMP threads the oracle will use (1 without OpenMP). */
int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
