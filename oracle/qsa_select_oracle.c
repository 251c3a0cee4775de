/*
 * qsa_select_oracle.c -- plain, slow, fp64 CPU oracle for the QSA route
 * producer (compressed-block index scores, top-k, expansion to token IDs).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the tests, the package-free smoke check and the CPU baseline
 * leg of the benchmark use it.  It shares no code, header, table or helper with
 * the CUDA library; the two meet only through the seeded input generator.
 *
 * What it computes follows the NeMo-AutoModel Qwen3.8-Flash-Next qsa page,
 * select_qsa_token_ids:
 *
 *   - query row t of batch b sits at global position tg = offset + t
 *     (query_position_offset: zero without context parallelism);
 *   - only the floor((tg + 1) / c) complete blocks are visible (c =
 *     compress_ratio);
 *   - a visible block's score is sum_h relu(dot(q[t,h], k[block])) / sqrt(D);
 *   - the best floor(token_budget / c) visible blocks are expanded to their c
 *     token IDs, and the tokens of the incomplete causal tail (0 .. c-1 of
 *     them, positions floor((tg + 1) / c) * c .. tg) are appended;
 *   - the row has token_budget + c - 1 slots; unused slots are -1.
 *
 * Readings where the page is silent (the same list is kept with the design
 * notes): IDs of a row are reported ascending (blocks ascending, then the
 * tail), so the row is already the sorted unique route set the attention path
 * builds; among blocks of equal score the lower block index wins; when no more
 * than floor(token_budget / c) blocks are visible all of them are taken (the
 * row is then dense causal); a row at or past its sequence's logical length
 * (sequence_lengths, right padding) has no routes: all -1.
 *
 * Layouts (all dense, row-major):
 *   q      : [B, S_q, H, D]          k : [B, NB, D]  (NB = floor(S_global / c))
 *   scores : [B, S_q, NB] double; invisible blocks hold -INFINITY
 *   seq_len: [B] int64               ids : [B, S_q, token_budget + c - 1] int32
 *
 * Return value of every entry point: 0 on success, -1 on a bad shape,
 * -2 when memory could not be allocated.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

typedef struct {
    int64_t B, S_q, H, D, NB, budget, c, offset;
} qsa_select_oracle_shape;

static int sel_shape_ok(const qsa_select_oracle_shape *s) {
    if (!s) return 0;
    if (s->B <= 0 || s->S_q <= 0 || s->H <= 0 || s->D <= 0 || s->NB < 0 || s->budget < 0 || s->c <= 0 ||
        s->offset < 0)
        return 0;
    /* every query position must lie inside the global sequence, which has NB complete blocks
     * and at most c - 1 further tokens */
    if (s->offset + s->S_q > s->NB * s->c + s->c - 1) return 0;
    if (s->NB * s->c > 2147483647LL) return 0; /* ids are reported as int32 */
    return 1;
}

/* Number of complete blocks visible from global position tg. */
static int64_t visible_blocks(int64_t tg, int64_t c) { return (tg + 1) / c; }

int qsa_oracle_index_scores(const qsa_select_oracle_shape *s, const double *q, const double *k, double *scores) {
    if (!sel_shape_ok(s) || !q || !k || !scores) return -1;
    const int64_t B = s->B, S_q = s->S_q, H = s->H, D = s->D, NB = s->NB;
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t b = 0; b < B; ++b)
        for (int64_t t = 0; t < S_q; ++t) {
            const int64_t nvis = visible_blocks(s->offset + t, s->c);
            double *row = scores + (b * S_q + t) * NB;
            for (int64_t blk = 0; blk < NB; ++blk) {
                if (blk >= nvis) {
                    row[blk] = -INFINITY;
                    continue;
                }
                const double *kb = k + (b * NB + blk) * D;
                double sum = 0.0;
                for (int64_t h = 0; h < H; ++h) {
                    const double *qh = q + ((b * S_q + t) * H + h) * D;
                    double dot = 0.0;
                    for (int64_t d = 0; d < D; ++d) dot += qh[d] * kb[d];
                    if (dot > 0.0) sum += dot; /* relu */
                }
                row[blk] = sum * inv_sqrt_d;
            }
        }
    return 0;
}

typedef struct {
    double score;
    int64_t blk;
} scored_block;

/* Best first: higher score, then lower block index. */
static int cmp_best_first(const void *a, const void *b) {
    const scored_block *x = (const scored_block *)a, *y = (const scored_block *)b;
    if (x->score != y->score) return x->score > y->score ? -1 : 1;
    return (x->blk > y->blk) - (x->blk < y->blk);
}

int qsa_oracle_select_ids(const qsa_select_oracle_shape *s, const double *scores, const int64_t *seq_len,
                          int32_t *ids) {
    if (!sel_shape_ok(s) || !scores || !seq_len || !ids) return -1;
    const int64_t B = s->B, S_q = s->S_q, NB = s->NB, c = s->c;
    const int64_t n_best = s->budget / c;
    const int64_t W = s->budget + c - 1;
    int err = 0;
#pragma omp parallel
    {
        scored_block *cand = (scored_block *)malloc((size_t)(NB > 0 ? NB : 1) * sizeof(scored_block));
        unsigned char *chosen = (unsigned char *)malloc((size_t)(NB > 0 ? NB : 1));
        if (!cand || !chosen) {
#pragma omp atomic write
            err = -2;
        }
#pragma omp for collapse(2) schedule(static)
        for (int64_t b = 0; b < B; ++b)
            for (int64_t t = 0; t < S_q; ++t) {
                if (!cand || !chosen) continue;
                int32_t *out = ids + (b * S_q + t) * W;
                const int64_t tg = s->offset + t;
                int64_t n = 0;
                if (tg < seq_len[b]) {
                    const int64_t nvis = visible_blocks(tg, c);
                    const double *row = scores + (b * S_q + t) * NB;
                    for (int64_t blk = 0; blk < nvis; ++blk) chosen[blk] = 0;
                    if (nvis <= n_best) {
                        for (int64_t blk = 0; blk < nvis; ++blk) chosen[blk] = 1;
                    } else {
                        for (int64_t blk = 0; blk < nvis; ++blk) {
                            cand[blk].score = row[blk];
                            cand[blk].blk = blk;
                        }
                        qsort(cand, (size_t)nvis, sizeof(scored_block), cmp_best_first);
                        for (int64_t i = 0; i < n_best; ++i) chosen[cand[i].blk] = 1;
                    }
                    for (int64_t blk = 0; blk < nvis; ++blk)
                        if (chosen[blk])
                            for (int64_t i = 0; i < c; ++i) out[n++] = (int32_t)(blk * c + i);
                    for (int64_t p = nvis * c; p <= tg; ++p) out[n++] = (int32_t)p; /* causal tail */
                }
                for (; n < W; ++n) out[n] = -1;
            }
        free(cand);
        free(chosen);
    }
    return err;
}
