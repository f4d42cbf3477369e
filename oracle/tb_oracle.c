/*
 * CPU oracle for the TokenButler decode-time hot path.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, fp64 statement of
 * what the decode path computes. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load it. It shares no code, header, table or
 * constant with the CUDA library; neither side includes or links the other.
 *
 * Sources (page title, then the section used):
 *   [abstract]  "TokenButler: Token Importance is Predictable", arXiv abstract
 *               (searcharxiv.com author page; fugumt.com v1 page).
 *   [summary]   "TokenButler: Token Importance is Predictable", gist.science
 *               technical summary, sections "Core Architecture",
 *               "Inference Strategy" and "Optimizations".
 *
 * Every array is dense and row-major. bf16 values travel as their raw 16-bit
 * patterns (uint16_t); a bf16 value widens to double exactly.
 *
 * Threads: OpenMP over independent (batch, KV head) rows. No step is blocked,
 * fused or reordered beyond what its definition states.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* bf16 <-> double                                                     */
/* ------------------------------------------------------------------ */

/* Exact widening: a bf16 pattern is the top half of an IEEE binary32. */
double tbo_bf16_to_double(uint16_t h)
{
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * Round a double to the nearest bf16 (8 significant bits, binary32 exponent
 * range), ties to even, in ONE rounding step (no detour through binary32,
 * which would round twice). Overflow goes to +-inf, NaN to the quiet NaN.
 */
uint16_t tbo_bf16_from_double(double x)
{
    if (isnan(x)) return 0x7FC0u;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);          /* a lies in [2^(e-1), 2^e) */
    int q = e - 8;               /* spacing of 8-significant-bit numbers there */
    if (q < -133) q = -133;      /* below 2^-126 the spacing is fixed at 2^-133 */
    double m = nearbyint(ldexp(a, -q));   /* default mode: nearest, ties to even */
    double v = ldexp(m, q);
    if (v >= 0x1p128) return (uint16_t)(sign | 0x7F80u);
    float f = (float)v;          /* exact: v has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

int tbo_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void tbo_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------ */
/* Step 1: key projection                                              */
/* ------------------------------------------------------------------ */

/*
 * [summary] Core Architecture, "Key-Cache Projection": each consumer layer
 * multiplies its full keys by a trained matrix into the low-dimensional
 * importance space. One matrix per KV head (Wk[h] is D x dp).
 *
 *   Kp64[b,h,t,j] = sum_d K[b,h,t,d] * Wk[h,d,j]       (fp64)
 *   Kp[b,h,t,j]   = RNE_bf16(Kp64[b,h,t,j])             (the cache stores bf16)
 *
 * K : [B, Hkv, n, D] bf16     Wk : [Hkv, D, dp] bf16
 * Kp: [B, Hkv, n, dp] bf16 out; Kp64 (may be NULL): same shape, fp64 out.
 */
void tbo_project(int B, int Hkv, int64_t n, int D, int dp,
                 const uint16_t *K, const uint16_t *Wk,
                 uint16_t *Kp, double *Kp64)
{
    #pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hkv; ++h) {
            const uint16_t *Kh = K + ((int64_t)b * Hkv + h) * n * D;
            const uint16_t *W = Wk + (int64_t)h * D * dp;
            uint16_t *Ph = Kp + ((int64_t)b * Hkv + h) * n * dp;
            double *P64 = Kp64 ? Kp64 + ((int64_t)b * Hkv + h) * n * dp : NULL;
            for (int64_t t = 0; t < n; ++t) {
                for (int j = 0; j < dp; ++j) {
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d)
                        acc += tbo_bf16_to_double(Kh[t * D + d]) *
                               tbo_bf16_to_double(W[(int64_t)d * dp + j]);
                    Ph[t * dp + j] = tbo_bf16_from_double(acc);
                    if (P64) P64[t * dp + j] = acc;
                }
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* Step 2: importance scores                                           */
/* ------------------------------------------------------------------ */

#define TBO_AGG_MEAN 0
#define TBO_AGG_MAX 1

/*
 * [abstract] the importance queries are combined with the projected keys to
 * score tokens; [summary] Core Architecture, "Scoring": a token's importance
 * is the inner product of a predicted query with the token's projected key.
 *
 * The G = Hq/Hkv query heads that share KV head h each carry their own
 * importance query; one budget is spent per KV head, so their G dot products
 * are aggregated: mean (agg = 0) or max (agg = 1).
 *
 *   s[b,h,t] = agg_{g<G} sum_i q_imp[b, h*G+g, i] * Kp[b,h,t,i]      (fp64)
 *
 * q_imp: [B, Hq, dp] bf16   Kp: [B, Hkv, n, dp] bf16   s: [B, Hkv, n] fp64 out
 * l1 (may be NULL): [B, Hkv, n] fp64 out, agg_g sum_i |q_imp * Kp| with the
 * same aggregation, the scale of the summation error bound.
 */
void tbo_score(int B, int Hq, int Hkv, int64_t n, int dp,
               const uint16_t *q_imp, const uint16_t *Kp, int agg,
               double *s, double *l1)
{
    int G = Hq / Hkv;
    #pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hkv; ++h) {
            const uint16_t *P = Kp + ((int64_t)b * Hkv + h) * n * dp;
            double *srow = s + ((int64_t)b * Hkv + h) * n;
            double *lrow = l1 ? l1 + ((int64_t)b * Hkv + h) * n : NULL;
            for (int64_t t = 0; t < n; ++t) {
                double best = -INFINITY, sum = 0.0, lbest = 0.0, lsum = 0.0;
                for (int g = 0; g < G; ++g) {
                    const uint16_t *qg = q_imp + ((int64_t)b * Hq + (int64_t)h * G + g) * dp;
                    double dot = 0.0, mag = 0.0;
                    for (int i = 0; i < dp; ++i) {
                        double p = tbo_bf16_to_double(qg[i]) *
                                   tbo_bf16_to_double(P[t * dp + i]);
                        dot += p;
                        mag += fabs(p);
                    }
                    sum += dot;
                    lsum += mag;
                    if (dot > best) best = dot;
                    if (mag > lbest) lbest = mag;
                }
                srow[t] = (agg == TBO_AGG_MAX) ? best : sum / G;
                if (lrow) lrow[t] = (agg == TBO_AGG_MAX) ? lbest : lsum / G;
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* Step 3: fixed-budget per-token top-k                                */
/* ------------------------------------------------------------------ */

typedef struct { double s; int32_t i; } tbo_pair;

/* Order: larger score first; among equal scores the lower index first.
 * -0.0 and +0.0 compare equal, so they tie and the index decides. */
static int tbo_pair_cmp(const void *pa, const void *pb)
{
    const tbo_pair *a = (const tbo_pair *)pa, *b = (const tbo_pair *)pb;
    if (a->s > b->s) return -1;
    if (a->s < b->s) return 1;
    return (a->i < b->i) ? -1 : (a->i > b->i);
}

static int tbo_int_cmp(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/*
 * [abstract] individual tokens are chosen, a fixed number k of them; [summary]
 * Core Architecture, Scoring. Per row (one (batch, KV head) pair) keep the k
 * tokens with the largest scores, ties to the lower index, and report their
 * indices in ascending order.
 *
 * s: [rows, n] fp64   idx: [rows, k] int32 out.
 * Returns 0, or -1 when a score is NaN (not an ordered value) or k is not in
 * [0, n].
 */
int tbo_topk(int64_t rows, int64_t n, int64_t k, const double *s, int32_t *idx)
{
    if (k < 0 || k > n) return -1;
    for (int64_t x = 0; x < rows * n; ++x)
        if (isnan(s[x])) return -1;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        tbo_pair *p = (tbo_pair *)malloc((size_t)(n > 0 ? n : 1) * sizeof *p);
        for (int64_t t = 0; t < n; ++t) { p[t].s = s[r * n + t]; p[t].i = (int32_t)t; }
        qsort(p, (size_t)n, sizeof *p, tbo_pair_cmp);
        int32_t *out = idx + r * k;
        for (int64_t j = 0; j < k; ++j) out[j] = p[j].i;
        qsort(out, (size_t)k, sizeof *out, tbo_int_cmp);
        free(p);
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Step 4: prediction interval and neighbour fetching                  */
/* ------------------------------------------------------------------ */

/*
 * [summary] Optimizations, "Prediction Interval & Neighbor Fetching": the
 * selection made at a prediction step is reused until the next one, and every
 * selected token brings the tokens next to it along.
 *
 * Reading used here: the prediction looked at the n_pred tokens present then;
 * each selected index i contributes [i-r, i+r] clipped to [0, n_pred); the
 * union is kept once, ascending; the tokens appended since the prediction,
 * [n_pred, n_t), follow it (they were never scored).
 *
 * idx: [rows, k] ascending   sel: [rows, sel_stride] out   counts: [rows] out
 * Returns 0, or -1 when a row would not fit in sel_stride or an index is out
 * of [0, n_pred).
 */
int tbo_expand(int64_t rows, int64_t k, const int32_t *idx, int r,
               int64_t n_pred, int64_t n_t, int32_t *sel, int64_t sel_stride,
               int32_t *counts)
{
    int bad = 0;
    unsigned char *mask = (unsigned char *)malloc((size_t)(n_pred > 0 ? n_pred : 1));
    for (int64_t row = 0; row < rows; ++row) {
        memset(mask, 0, (size_t)(n_pred > 0 ? n_pred : 1));
        for (int64_t j = 0; j < k; ++j) {
            int64_t i = idx[row * k + j];
            if (i < 0 || i >= n_pred) { bad = 1; continue; }
            for (int64_t t = i - r; t <= i + r; ++t)
                if (t >= 0 && t < n_pred) mask[t] = 1;
        }
        int64_t c = 0;
        for (int64_t t = 0; t < n_pred; ++t) {
            if (!mask[t]) continue;
            if (c < sel_stride) sel[row * sel_stride + c] = (int32_t)t;
            ++c;
        }
        for (int64_t t = n_pred; t < n_t; ++t) {
            if (c < sel_stride) sel[row * sel_stride + c] = (int32_t)t;
            ++c;
        }
        if (c > sel_stride) bad = 1;
        counts[row] = (int32_t)c;
    }
    free(mask);
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* Step 5: exact attention over the selected rows                      */
/* ------------------------------------------------------------------ */

/*
 * [abstract] the full KV cache is kept and only the selected tokens take part
 * in the step; [summary] Significance: only the relevant tokens are read.
 * Plain softmax attention of each query head over the selected rows of its
 * KV head:
 *
 *   z_j  = scale * sum_d q[b,hq,d] * K[b,h,j,d]             j in sel[b,h]
 *   w_j  = exp(z_j - max z) / sum_j' exp(z_j' - max z)
 *   out  = sum_j w_j * V[b,h,j,:]
 *
 * with h = hq / G. Everything in fp64.
 *
 * q: [B, Hq, D]   K, V: [B, Hkv, n_cache, D]   sel: [B, Hkv, sel_stride]
 * counts: [B, Hkv]   out: [B, Hq, D] fp64 out
 * wsum (may be NULL): [B, Hq] out, the sum of the weights w_j as computed.
 * Returns 0, or -1 for an index outside [0, n_cache) or an empty selection.
 */
int tbo_attn(int B, int Hq, int Hkv, int D, int64_t n_cache,
             const uint16_t *q, const uint16_t *K, const uint16_t *V,
             const int32_t *sel, const int32_t *counts, int64_t sel_stride,
             double scale, double *out, double *wsum)
{
    int G = Hq / Hkv;
    int bad = 0;
    #pragma omp parallel for collapse(2) schedule(dynamic, 1) reduction(|:bad)
    for (int b = 0; b < B; ++b) {
        for (int hq = 0; hq < Hq; ++hq) {
            int h = hq / G;
            const int32_t *srow = sel + ((int64_t)b * Hkv + h) * sel_stride;
            int64_t c = counts[(int64_t)b * Hkv + h];
            const uint16_t *qv = q + ((int64_t)b * Hq + hq) * D;
            const uint16_t *Kh = K + ((int64_t)b * Hkv + h) * n_cache * D;
            const uint16_t *Vh = V + ((int64_t)b * Hkv + h) * n_cache * D;
            double *o = out + ((int64_t)b * Hq + hq) * D;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            if (c <= 0) { bad = 1; continue; }
            double *z = (double *)malloc((size_t)c * sizeof *z);
            double zmax = -INFINITY;
            for (int64_t j = 0; j < c; ++j) {
                int64_t t = srow[j];
                if (t < 0 || t >= n_cache) { bad = 1; z[j] = -INFINITY; continue; }
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += tbo_bf16_to_double(qv[d]) * tbo_bf16_to_double(Kh[t * D + d]);
                z[j] = scale * dot;
                if (z[j] > zmax) zmax = z[j];
            }
            double denom = 0.0;
            for (int64_t j = 0; j < c; ++j) denom += exp(z[j] - zmax);
            double ws = 0.0;
            for (int64_t j = 0; j < c; ++j) {
                int64_t t = srow[j];
                if (t < 0 || t >= n_cache) continue;
                double w = exp(z[j] - zmax) / denom;
                ws += w;
                for (int d = 0; d < D; ++d)
                    o[d] += w * tbo_bf16_to_double(Vh[t * D + d]);
            }
            if (wsum) wsum[(int64_t)b * Hq + hq] = ws;
            free(z);
        }
    }
    return bad ? -1 : 0;
}
