/*
 * qsa_oracle.c -- plain, slow, fp64 CPU oracle for route-set sparse GQA attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the tests, the package-free smoke check and the CPU baseline
 * leg of the benchmark use it.  It shares no code, header, table or helper with
 * the CUDA library; the two meet only through the seeded input generator.
 *
 * What it computes is the plain definition of "exact route-set GQA" as the
 * NeMo-AutoModel Qwen3.8-Flash-Next pages state it:
 *
 *   - flex_qsa, module docstring: every layout reduces to "each query row
 *     attends exactly to its route IDs"; rows whose routes are all -1 give
 *     exactly zero output and zero gradients.
 *   - flex_qsa, _routes_to_membership / flex_sparse_gqa_attention parameters:
 *     negative or out-of-range entries are padding.
 *   - fa4_qsa, _preprocess: duplicate IDs collapse; invalid IDs, large int64
 *     values included, are discarded before indexing.
 *   - fa4_qsa, fa4_sparse_gqa_attention: no triangular mask is added (routes
 *     encode causality); query_heads is a positive multiple of kv_heads.
 *   - qsa, _gathered_qsa_gqa_attention_chunk: queries are grouped as
 *     [B, Q, Hkv, G, D], so query head h reads KV head floor(h / G).
 *   - flex_sparse_gqa_attention: the score multiplier defaults to 1/sqrt(D)
 *     (resolved by the caller; this file takes the scale as given).
 *
 * Readings where the pages are silent (the same list is kept with the design
 * notes): LSE is the natural log of sum_j exp(scaled score), stored [B,Hq,S_q],
 * -inf for an empty row; the deduplicated IDs are reported ascending; Delta in
 * the backward pass is sum_j P_j dP_j; an empty row contributes nothing to
 * dK/dV.
 *
 * Every accumulation is in double.  There is no blocking, fusion or reordering
 * beyond the definition; OpenMP only splits independent rows (or keys) across
 * threads, and every sum is taken in one fixed order, so results do not depend
 * on the thread count.
 *
 * Layouts (all dense, row-major):
 *   q, o, dout, dq : [B, S_q, Hq, D]        k, v : [B, S_kv, Hkv, D]
 *   routes         : [B, S_q, K] int64       lse  : [B, Hq, S_q]
 *   ids            : [B, S_q, K] int32 (ascending unique valid IDs, then -1)
 *   counts         : [B, S_q] int32
 *   dk, dv         : [B, S_kv, Hkv, D], or [n_keys, Hkv, D] when a key list
 *                    (flat b * S_kv + j) is given.
 *
 * Return value of every entry point: 0 on success, -1 on a bad shape,
 * -2 when memory could not be allocated.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t B, S_q, S_kv, Hq, Hkv, D, K;
} qsa_oracle_shape;

static int shape_ok(const qsa_oracle_shape *s) {
    if (!s) return 0;
    if (s->B <= 0 || s->S_q <= 0 || s->S_kv <= 0 || s->Hq <= 0 || s->Hkv <= 0 || s->D <= 0 || s->K <= 0)
        return 0;
    if (s->Hq % s->Hkv != 0) return 0;
    if (s->S_kv > 2147483647LL) return 0; /* ids are reported as int32 */
    return 1;
}

static int cmp_i64(const void *a, const void *b) {
    int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
    return (x > y) - (x < y);
}

/* Route set of one row: the valid entries (0 <= id < S_kv, compared in int64
 * before any narrowing), sorted ascending, repeats dropped.  Writes up to K
 * ids into out and returns how many. */
static int64_t row_route_set(const int64_t *row, int64_t K, int64_t S_kv, int64_t *tmp, int32_t *out) {
    int64_t n = 0;
    for (int64_t k = 0; k < K; ++k) {
        int64_t x = row[k];
        if (x >= 0 && x < S_kv) tmp[n++] = x;
    }
    qsort(tmp, (size_t)n, sizeof(int64_t), cmp_i64);
    int64_t u = 0;
    for (int64_t i = 0; i < n; ++i)
        if (i == 0 || tmp[i] != tmp[i - 1]) out[u++] = (int32_t)tmp[i];
    return u;
}

int qsa_oracle_route_sets(const qsa_oracle_shape *s, const int64_t *routes, int32_t *ids, int32_t *counts) {
    if (!shape_ok(s) || !routes || !ids || !counts) return -1;
    const int64_t rows = s->B * s->S_q, K = s->K;
    int err = 0;
#pragma omp parallel
    {
        int64_t *tmp = (int64_t *)malloc((size_t)K * sizeof(int64_t));
        if (!tmp) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 64)
        for (int64_t r = 0; r < rows; ++r) {
            if (!tmp) continue;
            int32_t *out = ids + r * K;
            int64_t n = row_route_set(routes + r * K, K, s->S_kv, tmp, out);
            for (int64_t i = n; i < K; ++i) out[i] = -1;
            counts[r] = (int32_t)n;
        }
        free(tmp);
    }
    return err;
}

/* Route sets for every row, computed once per call. */
static int all_route_sets(const qsa_oracle_shape *s, const int64_t *routes, int32_t **ids, int32_t **counts) {
    const int64_t rows = s->B * s->S_q;
    *ids = (int32_t *)malloc((size_t)(rows * s->K) * sizeof(int32_t));
    *counts = (int32_t *)malloc((size_t)rows * sizeof(int32_t));
    if (!*ids || !*counts) {
        free(*ids);
        free(*counts);
        return -2;
    }
    return qsa_oracle_route_sets(s, routes, *ids, *counts);
}

static double dot(const double *a, const double *b, int64_t n) {
    double acc = 0.0;
    for (int64_t i = 0; i < n; ++i) acc += a[i] * b[i];
    return acc;
}

/* Softmax of one (row, head) over its route set R (n entries):
 *   s_j = scale * <q_h, k_j>,  m = max_j s_j,  l = sum_j exp(s_j - m),
 *   P_j = exp(s_j - m) / l,    LSE = m + ln l.
 * Fills p[0..n) and returns LSE.  n must be positive. */
static double row_softmax(const double *qh, const double *kbase, int64_t kstride, const int32_t *R, int64_t n,
                          int64_t D, double scale, double *p) {
    double m = -INFINITY;
    for (int64_t t = 0; t < n; ++t) {
        p[t] = scale * dot(qh, kbase + (int64_t)R[t] * kstride, D);
        if (p[t] > m) m = p[t];
    }
    double l = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        p[t] = exp(p[t] - m);
        l += p[t];
    }
    for (int64_t t = 0; t < n; ++t) p[t] /= l;
    return m + log(l);
}

int qsa_oracle_forward(const qsa_oracle_shape *s, const double *q, const double *k, const double *v,
                       const int64_t *routes, double scale, double *o, double *lse) {
    if (!shape_ok(s) || !q || !k || !v || !routes || !o || !lse) return -1;
    const int64_t B = s->B, S_q = s->S_q, S_kv = s->S_kv, Hq = s->Hq, Hkv = s->Hkv, D = s->D, K = s->K;
    const int64_t G = Hq / Hkv;
    int32_t *ids = NULL, *counts = NULL;
    int rc = all_route_sets(s, routes, &ids, &counts);
    if (rc) return rc;
    int err = 0;
#pragma omp parallel
    {
        double *p = (double *)malloc((size_t)K * sizeof(double));
        if (!p) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < B * S_q; ++r) {
            if (!p) continue;
            const int64_t b = r / S_q, qi = r % S_q;
            const int32_t *R = ids + r * K;
            const int64_t n = counts[r];
            for (int64_t h = 0; h < Hq; ++h) {
                const int64_t g = h / G;
                const double *qh = q + (r * Hq + h) * D;
                double *oh = o + (r * Hq + h) * D;
                double *lse_h = lse + (b * Hq + h) * S_q + qi;
                for (int64_t d = 0; d < D; ++d) oh[d] = 0.0;
                if (n == 0) { /* empty route set: zero output, LSE = -inf */
                    *lse_h = -INFINITY;
                    continue;
                }
                const double *kb = k + (b * S_kv * Hkv + g) * D;
                const double *vb = v + (b * S_kv * Hkv + g) * D;
                *lse_h = row_softmax(qh, kb, Hkv * D, R, n, D, scale, p);
                for (int64_t t = 0; t < n; ++t) {
                    const double *vj = vb + (int64_t)R[t] * Hkv * D;
                    for (int64_t d = 0; d < D; ++d) oh[d] += p[t] * vj[d];
                }
            }
        }
        free(p);
    }
    free(ids);
    free(counts);
    return err;
}

static int in_sorted(const int32_t *R, int64_t n, int64_t x) {
    int64_t lo = 0, hi = n;
    while (lo < hi) {
        int64_t mid = (lo + hi) / 2;
        if (R[mid] < x) lo = mid + 1;
        else hi = mid;
    }
    return lo < n && R[lo] == x;
}

/* First-order backward by the direct formulas, given dout = dL/dO:
 *   dP_j  = <dO_h, v_j>,     Delta = sum_j P_j dP_j,    dS_j = P_j (dP_j - Delta),
 *   dQ_h  = scale * sum_j dS_j k_j,
 *   dK_j += scale * dS_j q_h,  dV_j += P_j dO_h   (summed over every row and
 *   every head h of the KV head's group that routes to j).
 * dq is always computed for every row.  dK/dV are computed for every key when
 * keys == NULL, else only for the n_keys listed keys (flat b * S_kv + j); each
 * key's sum runs over rows in ascending order, heads ascending, so a listed key
 * gets exactly the value the full computation gives it. */
int qsa_oracle_backward(const qsa_oracle_shape *s, const double *q, const double *k, const double *v,
                        const int64_t *routes, const double *dout, double scale, double *dq, int64_t n_keys,
                        const int64_t *keys, double *dk, double *dv) {
    if (!shape_ok(s) || !q || !k || !v || !routes || !dout || !dq || !dk || !dv) return -1;
    const int64_t B = s->B, S_q = s->S_q, S_kv = s->S_kv, Hq = s->Hq, Hkv = s->Hkv, D = s->D, K = s->K;
    const int64_t G = Hq / Hkv;
    const int64_t rows = B * S_q;
    if (keys) {
        if (n_keys < 0) return -1;
        for (int64_t i = 0; i < n_keys; ++i)
            if (keys[i] < 0 || keys[i] >= B * S_kv) return -1;
    } else {
        n_keys = B * S_kv;
    }
    int32_t *ids = NULL, *counts = NULL;
    int rc = all_route_sets(s, routes, &ids, &counts);
    if (rc) return rc;
    /* Per (row, head): LSE and Delta, needed to rebuild P_j and dS_j of a
     * single key in the dK/dV pass. */
    double *row_lse = (double *)malloc((size_t)(rows * Hq) * sizeof(double));
    double *row_delta = (double *)malloc((size_t)(rows * Hq) * sizeof(double));
    if (!row_lse || !row_delta) {
        free(row_lse);
        free(row_delta);
        free(ids);
        free(counts);
        return -2;
    }
    int err = 0;
#pragma omp parallel
    {
        double *p = (double *)malloc((size_t)K * sizeof(double));
        double *dp = (double *)malloc((size_t)K * sizeof(double));
        if (!p || !dp) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < rows; ++r) {
            if (!p || !dp) continue;
            const int64_t b = r / S_q;
            const int32_t *R = ids + r * K;
            const int64_t n = counts[r];
            for (int64_t h = 0; h < Hq; ++h) {
                const int64_t g = h / G;
                const double *qh = q + (r * Hq + h) * D;
                const double *doh = dout + (r * Hq + h) * D;
                double *dqh = dq + (r * Hq + h) * D;
                for (int64_t d = 0; d < D; ++d) dqh[d] = 0.0;
                if (n == 0) { /* empty row: zero query gradient, no dK/dV term */
                    row_lse[r * Hq + h] = -INFINITY;
                    row_delta[r * Hq + h] = 0.0;
                    continue;
                }
                const double *kb = k + (b * S_kv * Hkv + g) * D;
                const double *vb = v + (b * S_kv * Hkv + g) * D;
                row_lse[r * Hq + h] = row_softmax(qh, kb, Hkv * D, R, n, D, scale, p);
                double delta = 0.0;
                for (int64_t t = 0; t < n; ++t) {
                    dp[t] = dot(doh, vb + (int64_t)R[t] * Hkv * D, D);
                    delta += p[t] * dp[t];
                }
                row_delta[r * Hq + h] = delta;
                for (int64_t t = 0; t < n; ++t) {
                    const double ds = p[t] * (dp[t] - delta);
                    const double *kj = kb + (int64_t)R[t] * Hkv * D;
                    for (int64_t d = 0; d < D; ++d) dqh[d] += scale * ds * kj[d];
                }
            }
        }
        free(p);
        free(dp);
    }
    if (err) goto done;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < n_keys; ++i) {
        const int64_t flat = keys ? keys[i] : i;
        const int64_t b = flat / S_kv, j = flat % S_kv;
        for (int64_t g = 0; g < Hkv; ++g) {
            double *dkj = dk + (i * Hkv + g) * D;
            double *dvj = dv + (i * Hkv + g) * D;
            for (int64_t d = 0; d < D; ++d) dkj[d] = dvj[d] = 0.0;
            const double *kj = k + ((b * S_kv + j) * Hkv + g) * D;
            const double *vj = v + ((b * S_kv + j) * Hkv + g) * D;
            for (int64_t qi = 0; qi < S_q; ++qi) {
                const int64_t r = b * S_q + qi;
                if (!in_sorted(ids + r * K, counts[r], j)) continue;
                for (int64_t h = g * G; h < (g + 1) * G; ++h) {
                    const double *qh = q + (r * Hq + h) * D;
                    const double *doh = dout + (r * Hq + h) * D;
                    const double pj = exp(scale * dot(qh, kj, D) - row_lse[r * Hq + h]);
                    const double ds = pj * (dot(doh, vj, D) - row_delta[r * Hq + h]);
                    for (int64_t d = 0; d < D; ++d) {
                        dkj[d] += scale * ds * qh[d];
                        dvj[d] += pj * doh[d];
                    }
                }
            }
        }
    }
done:
    free(row_lse);
    free(row_delta);
    free(ids);
    free(counts);
    return err;
}
