/*
 * oracle.c -- plain, slow, fp64 CPU oracle of the KV-cache eviction path.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg call this code; the product path never does.
 * It shares no code, header or constant with the CUDA library.
 *
 * What it computes, for one unit = (request, layer, KV head) with n cached
 * tokens, head dim d, a GQA group of G query heads and an observation window
 * of the last w query positions (R = G*w query rows):
 *
 *  1. Window attention (DropKV, "Methodology in Plain English": the attention
 *     output a the removal shift is measured against).  Row i = g*w + t is
 *     query head g of the group at position pos = n - w + t; it attends
 *     causally to keys 0..pos with logits s_j = scale * <q, k_j>,
 *     p_j = exp(s_j - max) / sum_i exp(s_i - max), a = sum_j p_j v_j.
 *
 *  2. Removal score (DropKV, "Key Contributions" item 1 and "Methodology in
 *     Plain English"): deleting token j alone shifts the output by
 *     p_j / (1 - p_j) * ||a - v_j||_2.  The per-token score is that shift
 *     summed, without squaring, over the R rows that see token j.  The
 *     norm is taken directly on the difference vector, not by expansion.
 *
 *  3. Selection (DropKV "Methodology": keep the highest-scoring tokens, pin
 *     the most recent w; PyramidKV blog, "Observation Window and Aggregated
 *     Attention Eviction": keep the first 4 sink tokens, the top tokens and
 *     the recent window).  The budget b counts sinks and window; the middle
 *     candidates [sinks, n-w) are ranked by (score descending, index
 *     ascending) and the first b - sinks - w kept.  Output: ascending indices.
 *
 * All arithmetic is IEEE double; inputs are bfloat16 bit patterns, widened
 * exactly.  Compile with -ffp-contract=off so no step is fused.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* logits of one query row against keys 0..pos, into s[0..pos]; returns their max */
static double row_logits(int pos, int d, double scale, const uint16_t *qrow,
                         const uint16_t *k, double *s) {
    double mx = -INFINITY;
    for (int j = 0; j <= pos; ++j) {
        const uint16_t *kj = k + (size_t)j * d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += bf16_value(qrow[c]) * bf16_value(kj[c]);
        s[j] = scale * dot;
        if (s[j] > mx) mx = s[j];
    }
    return mx;
}

/*
 * Window attention of one unit.
 *   q: [G*w][d] bf16 bits (row i = head g*w + window slot t)
 *   k, v: [n][d] bf16 bits
 *   out m[R] (row max of the logits), l[R] (sum of exp(s - m)), a[R][d].
 * Returns 0, or -1 on bad sizes / allocation failure.
 */
int oracle_window_attention(int n, int d, int G, int w, double scale,
                            const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            double *m, double *l, double *a) {
    if (n < 1 || d < 1 || G < 1 || w < 1 || w > n) return -1;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    if (!s) return -1;
    const int R = G * w;
    for (int i = 0; i < R; ++i) {
        const int pos = n - w + (i % w);
        const uint16_t *qrow = q + (size_t)i * d;
        const double mx = row_logits(pos, d, scale, qrow, k, s);
        double sum = 0.0;
        for (int j = 0; j <= pos; ++j) {
            s[j] = exp(s[j] - mx);
            sum += s[j];
        }
        double *ai = a + (size_t)i * d;
        for (int c = 0; c < d; ++c) ai[c] = 0.0;
        for (int j = 0; j <= pos; ++j) {
            const double p = s[j] / sum;
            const uint16_t *vj = v + (size_t)j * d;
            for (int c = 0; c < d; ++c) ai[c] += p * bf16_value(vj[c]);
        }
        m[i] = mx;
        l[i] = sum;
    }
    free(s);
    return 0;
}

/*
 * Removal scores of one unit: S[j] = sum over rows i that see j of
 *   p_ij / (1 - p_ij) * || a_i - v_j ||_2.
 * Returns 0; -1 on bad sizes / allocation failure; -2 if some p_ij == 1
 * (a row that sees a single key: the shift of deleting it is unbounded).
 */
int oracle_unit_scores(int n, int d, int G, int w, double scale,
                       const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       double *S) {
    if (n < 1 || d < 1 || G < 1 || w < 1 || w > n) return -1;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double *a = (double *)malloc(sizeof(double) * (size_t)d);
    if (!s || !a) { free(s); free(a); return -1; }
    for (int j = 0; j < n; ++j) S[j] = 0.0;
    const int R = G * w;
    int rc = 0;
    for (int i = 0; i < R && rc == 0; ++i) {
        const int pos = n - w + (i % w);
        const uint16_t *qrow = q + (size_t)i * d;
        const double mx = row_logits(pos, d, scale, qrow, k, s);
        double sum = 0.0;
        for (int j = 0; j <= pos; ++j) {
            s[j] = exp(s[j] - mx);
            sum += s[j];
        }
        for (int c = 0; c < d; ++c) a[c] = 0.0;
        for (int j = 0; j <= pos; ++j) {
            const double p = s[j] / sum;
            const uint16_t *vj = v + (size_t)j * d;
            for (int c = 0; c < d; ++c) a[c] += p * bf16_value(vj[c]);
        }
        for (int j = 0; j <= pos; ++j) {
            const double p = s[j] / sum;
            if (!(p < 1.0)) { rc = -2; break; }
            const uint16_t *vj = v + (size_t)j * d;
            double dist2 = 0.0;
            for (int c = 0; c < d; ++c) {
                const double diff = a[c] - bf16_value(vj[c]);
                dist2 += diff * diff;
            }
            S[j] += p / (1.0 - p) * sqrt(dist2);
        }
    }
    free(s);
    free(a);
    return rc;
}

/*
 * The other aggregation rules of one unit, over the same rows and keys as
 * oracle_unit_scores (row i sees keys 0..n-w+(i%w)):
 *   rule 1, squared (DropKV "Methodology in Plain English": the per-token
 *     shift accumulated over the observation window and squared):
 *       S[j] = sum_i (p_ij / (1 - p_ij))^2 * ||a_i - v_j||_2^2
 *   rule 2, attention sum (PyramidKV guide, "Observation Window and
 *     Aggregated Attention Eviction": the attention weights of the window
 *     queries summed over queries and heads):
 *       S[j] = sum_i p_ij
 * Returns 0; -1 on bad sizes, rule or allocation failure; -2 if rule 1 meets
 * some p_ij == 1.
 */
int oracle_unit_scores_rule(int n, int d, int G, int w, double scale, int rule,
                            const uint16_t *q, const uint16_t *k, const uint16_t *v,
                            double *S) {
    if (n < 1 || d < 1 || G < 1 || w < 1 || w > n || rule < 1 || rule > 2) return -1;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double *a = (double *)malloc(sizeof(double) * (size_t)d);
    if (!s || !a) { free(s); free(a); return -1; }
    for (int j = 0; j < n; ++j) S[j] = 0.0;
    const int R = G * w;
    int rc = 0;
    for (int i = 0; i < R && rc == 0; ++i) {
        const int pos = n - w + (i % w);
        const uint16_t *qrow = q + (size_t)i * d;
        const double mx = row_logits(pos, d, scale, qrow, k, s);
        double sum = 0.0;
        for (int j = 0; j <= pos; ++j) {
            s[j] = exp(s[j] - mx);
            sum += s[j];
        }
        if (rule == 2) {
            for (int j = 0; j <= pos; ++j) S[j] += s[j] / sum;
            continue;
        }
        for (int c = 0; c < d; ++c) a[c] = 0.0;
        for (int j = 0; j <= pos; ++j) {
            const double p = s[j] / sum;
            const uint16_t *vj = v + (size_t)j * d;
            for (int c = 0; c < d; ++c) a[c] += p * bf16_value(vj[c]);
        }
        for (int j = 0; j <= pos; ++j) {
            const double p = s[j] / sum;
            if (!(p < 1.0)) { rc = -2; break; }
            const uint16_t *vj = v + (size_t)j * d;
            double dist2 = 0.0;
            for (int c = 0; c < d; ++c) {
                const double diff = a[c] - bf16_value(vj[c]);
                dist2 += diff * diff;
            }
            const double r = p / (1.0 - p);
            S[j] += r * r * dist2;
        }
    }
    free(s);
    free(a);
    return rc;
}

/*
 * Max pooling of one unit's scores (DropKV page: "a max-pool over neighbouring
 * scores", kernel size 11; BellowsKV blog: each token takes the maximum score
 * in a 13-position window centred on it): out[j] = max S[i] over
 * i in [j - r, j + r] within [0, n), r = (kernel - 1) / 2.  kernel must be odd.
 * Returns 0; -1 on bad sizes.
 */
int oracle_max_pool(int n, int kernel, const double *S, double *out) {
    if (n < 1 || kernel < 1 || kernel % 2 == 0) return -1;
    const int r = (kernel - 1) / 2;
    for (int j = 0; j < n; ++j) {
        double mx = -INFINITY;
        for (int i = j - r; i <= j + r; ++i)
            if (i >= 0 && i < n && S[i] > mx) mx = S[i];
        out[j] = mx;
    }
    return 0;
}

typedef struct { double score; int32_t idx; } ranked;

static int rank_cmp(const void *x, const void *y) {
    const ranked *a = (const ranked *)x, *b = (const ranked *)y;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->idx > b->idx) - (a->idx < b->idx);
}

/*
 * Budgeted selection of one unit.
 *   S[n] scores, b budget (sinks and window included).
 *   idx[b] out: kept token indices, ascending.
 * Returns 0; -1 if the sizes are inconsistent (needs sinks + w <= b <= n).
 */
int oracle_select(int n, int w, int sinks, int b, const double *S, int32_t *idx) {
    if (n < 1 || w < 0 || sinks < 0 || sinks + w > n || b < sinks + w || b > n) return -1;
    const int lo = sinks, hi = n - w;         /* middle candidates [lo, hi) */
    const int take = b - sinks - w;
    const int cnt = hi - lo;
    ranked *r = (ranked *)malloc(sizeof(ranked) * (size_t)(cnt > 0 ? cnt : 1));
    unsigned char *keep = (unsigned char *)calloc((size_t)n, 1);
    if (!r || !keep) { free(r); free(keep); return -1; }
    for (int j = lo; j < hi; ++j) { r[j - lo].score = S[j]; r[j - lo].idx = j; }
    qsort(r, (size_t)cnt, sizeof(ranked), rank_cmp);
    for (int j = 0; j < sinks; ++j) keep[j] = 1;
    for (int j = hi; j < n; ++j) keep[j] = 1;
    for (int t = 0; t < take; ++t) keep[r[t].idx] = 1;
    int o = 0;
    for (int j = 0; j < n; ++j)
        if (keep[j]) idx[o++] = j;
    free(r);
    free(keep);
    return o == b ? 0 : -1;
}
