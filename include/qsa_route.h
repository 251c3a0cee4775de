/*
 * qsa_route.h -- C ABI of the QSA route producer in libqsa.so: compressed-block
 * index scores, top-k block selection and expansion to token IDs, emitting the
 * route rows that qsa_preprocess / qsa_forward / qsa_backward (qsa.h) consume.
 *
 * The operation is select_qsa_token_ids of the NeMo-AutoModel
 * Qwen3.8-Flash-Next qsa page.  With c = compress_ratio, row t of batch b at
 * global position tg = query_position_offset + t:
 *
 *   nvis(tg)       = floor((tg + 1) / c)   complete blocks visible from tg
 *   score(t, blk)  = sum_h relu(<Qi[b,t,h,:], Kc[b,blk,:]>) / sqrt(D_index),  blk < nvis
 *   chosen(t)      = the floor(token_budget / c) visible blocks of highest score
 *                    (all visible blocks when there are no more than that)
 *   ids[b,t,:]     = the c token IDs of every chosen block, then the tokens
 *                    nvis*c .. tg of the incomplete causal tail (0 .. c-1 of
 *                    them), then -1, in a row of W = token_budget + c - 1 slots.
 *
 * Readings of points the page leaves open (the library's contract):
 *   - IDs are written ascending (chosen blocks ascending, then the tail), so
 *     every row already is the sorted, duplicate-free route set of qsa.h;
 *   - among blocks of equal score the lower block index is chosen;
 *   - a row with tg >= sequence_lengths[b] (right padding) is all -1;
 *   - scores are formed in fp32 from the BF16 inputs (fp32 accumulation, the
 *     relu-sum in fp32, times the fp32-rounded 1/sqrt(D_index)) and the
 *     selection compares those fp32 values exactly; +0 and -0 are equal;
 *     scores must not be NaN.
 * The page scores query rows in chunks only to bound a temporary score
 * tensor; the choice does not depend on chunking, and this library takes the
 * whole problem in one call (a caller may still split query rows into calls
 * with adjusted query_position_offset and pointers).
 *
 * Conventions are those of qsa.h: device pointers unless named *_host, caller
 * owns all memory, work is queued on `stream` with no host synchronisation,
 * errors are returned (no fallback), qsa_last_error() explains the last one,
 * and index arithmetic is 64-bit.  The workspace needs no initialisation:
 * every call that scores clears its status word and work queue counters
 * first; qsa_read_device_status(workspace) then reports (and clears) a
 * device-side failure of that call, such as a bounded wait that gave up
 * (QSA_ERR_TIMEOUT).  Calls sharing one workspace must be ordered.
 */
#ifndef QSA_ROUTE_H_
#define QSA_ROUTE_H_

#include "qsa.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Problem description (select_qsa_token_ids parameters):
 *   index_queries   : [B, S_q, H_index, D_index] BF16, strides q_stride (elements)
 *   compressed_keys : [B, n_blocks, D_index] BF16 (the page's [B, n_blocks, 1,
 *                     D_index] with the unit head dimension dropped), strides
 *                     k_stride (elements)
 *   sequence_lengths: [B] int64 logical lengths (right padding), device
 *   ids             : [B, S_q, token_budget + compress_ratio - 1] int32, dense
 * n_blocks = floor(S_global / compress_ratio) for the padded global length
 * S_global (S_q without context parallelism); query_position_offset is the
 * global position of local row 0 (cp_rank * S_q for the contiguous layout).
 * Every local position must lie inside the global sequence:
 * query_position_offset + S_q <= n_blocks * compress_ratio + compress_ratio - 1.
 * Supported: H_index a power of two, 1..128; D_index 64 or 128; token IDs and
 * the row width within int32; unit last strides, other strides multiples of 8
 * elements, 16-byte aligned bases. */
typedef struct qsa_route_problem {
    int64_t B, S_q, H_index, D_index, n_blocks;
    int64_t token_budget, compress_ratio, query_position_offset;
    int64_t q_stride[4];
    int64_t k_stride[3];
} qsa_route_problem;

/* Validates a route problem without touching the device. */
QSA_API qsa_status qsa_route_check_problem(const qsa_route_problem *problem);

/* Slots per output row: token_budget + compress_ratio - 1 (0 if invalid). */
QSA_API int64_t qsa_route_width(const qsa_route_problem *problem);

/* Bytes of device workspace qsa_select_token_ids needs (256-byte aligned base):
 * a status word, work queue counters and the fp32 score tensor
 * [B, S_q, n_blocks].  qsa_index_scores and qsa_select_from_scores need only the
 * first 512 bytes of it.  0 if the problem is invalid. */
QSA_API size_t qsa_route_workspace_bytes(const qsa_route_problem *problem);

/* Block scores alone: writes scores[(b * S_q + t) * n_blocks + blk] (fp32) for
 * every row with tg < sequence_lengths[b] and every blk < nvis(tg); other
 * entries are left as they were.  Tensor-core kernel (tcgen05, TMA). */
QSA_API qsa_status qsa_index_scores(const qsa_route_problem *problem, const void *index_queries,
                                    const void *compressed_keys, const int64_t *sequence_lengths, void *workspace,
                                    size_t ws_bytes, float *scores, cudaStream_t stream);

/* Selection and expansion alone, from scores laid out as qsa_index_scores
 * writes them (only the visible entries of live rows are read).  Writes every
 * slot of ids. */
QSA_API qsa_status qsa_select_from_scores(const qsa_route_problem *problem, const float *scores,
                                          const int64_t *sequence_lengths, void *workspace, size_t ws_bytes,
                                          int32_t *ids, cudaStream_t stream);

/* The route producer end to end (select_qsa_token_ids): scores into the
 * workspace, then selection into ids.  ids must not overlap the inputs or the
 * workspace. */
QSA_API qsa_status qsa_select_token_ids(const qsa_route_problem *problem, const void *index_queries,
                                        const void *compressed_keys, const int64_t *sequence_lengths,
                                        void *workspace, size_t ws_bytes, int32_t *ids, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QSA_ROUTE_H_ */
