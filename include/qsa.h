/*
 * qsa.h -- C ABI of the GB300 route-set sparse GQA attention library (libqsa.so).
 *
 * The operation is exact route-set grouped-query attention as the NeMo-AutoModel
 * Qwen3.8-Flash-Next pages define it (flex_qsa module docstring and
 * flex_sparse_gqa_attention; fa4_qsa fa4_sparse_gqa_attention and _preprocess;
 * qsa _gathered_qsa_gqa_attention_chunk):
 *
 *   for every batch b, query row q and query head h (KV head g = h / (Hq/Hkv)):
 *     R(b,q)  = the distinct route IDs x of row (b,q) with 0 <= x < S_kv
 *     s_j     = scale * <Q[b,q,h,:], K[b,j,g,:]>            for j in R(b,q)
 *     O[b,q,h,:] = sum_j softmax(s)_j * V[b,j,g,:],   LSE[b,h,q] = ln sum_j exp(s_j)
 *   An empty R gives O = 0, LSE = -inf, zero dQ and no dK/dV contribution.  No
 *   causal mask is added: routes alone encode causality, documents and padding.
 *
 * Conventions shared by every entry point
 *   - Pointers named q, k, v, o, dout, dq, dk, dv, lse, routes and workspace
 *     are DEVICE pointers on the current CUDA device; *_host pointers are host.
 *   - The caller owns every buffer.  No entry point allocates or frees device
 *     memory; the only device memory the library holds is the fixed array of
 *     qsa_forward_no_alloc (below).  Between calls it keeps no state about
 *     problems, only, per device, which kernels' shared-memory limits it has
 *     already raised.
 *   - All device work is queued on `stream`; no entry point blocks the host
 *     except qsa_read_device_status, which says so.
 *   - BF16 tensors are passed as `const void*` holding IEEE bfloat16 values.
 *   - Errors are returned, never silently worked around: there is no CPU or
 *     alternative-kernel fallback for an input the library rejects.
 *     qsa_last_error() gives a one-line reason for the last non-QSA_OK status
 *     returned on the calling host thread.
 *   - Invalid route VALUES (-1, other negatives, >= S_kv, huge int64) are not
 *     errors: they are padding (flex_qsa _routes_to_membership).
 *   - Index arithmetic is 64-bit throughout; B*S_q*S_kv may exceed 2^32
 *     (flex_qsa _membership_flat_offset explains the int32 wrap this avoids).
 */
#ifndef QSA_H_
#define QSA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define QSA_API __attribute__((visibility("default")))
#else
#define QSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum qsa_status {
    QSA_OK = 0,
    QSA_ERR_INVALID_ARGUMENT = 1,    /* empty dim, Hq % Hkv != 0, bad scale, null or aliasing pointer, bad route_bits */
    QSA_ERR_UNSUPPORTED = 2,         /* D not 64/128/256, S_kv > 2^31 - 1, K > 16384, non-unit last stride, misaligned */
    QSA_ERR_WORKSPACE_TOO_SMALL = 3, /* ws_bytes < qsa_workspace_bytes(problem) */
    QSA_ERR_CUDA = 4,                /* a CUDA runtime call or kernel launch failed */
    QSA_ERR_TIMEOUT = 5,             /* a device-side wait hit its iteration limit (reported by qsa_read_device_status) */
    QSA_ERR_DEVICE_CHECK = 6         /* a device-side bounds check fired (reported by qsa_read_device_status) */
} qsa_status;

/* Problem description.  Shapes follow flex_sparse_gqa_attention /
 * fa4_sparse_gqa_attention:
 *   Q, O, dO, dQ : [B, S_q, Hq, D]      K, V, dK, dV : [B, S_kv, Hkv, D]
 *   routes       : [B, S_q, K] signed int32 or int64 (route_bits = 32 or 64)
 *   LSE          : [B, Hq, S_q] float32, natural log
 * Hq must be a positive multiple of Hkv.  D is 256 as fa4_sparse_gqa_attention
 * fixes head_dim = 256 (the tensor-core tile kernels); D = 128 is also
 * accepted (tile kernels when G = Hq/Hkv is a power of two from 4 to 64, as at
 * D = 256; other G on warp-level kernels) and D = 64 runs on the warp-level
 * kernels.  S_kv may differ from S_q (context parallelism: local
 * queries against gathered global K/V).  softmax_scale must be finite and > 0;
 * the pages' default 1/sqrt(D) is resolved by the caller.
 * Strides are in elements.  q/k/v need a unit last stride and, for the other
 * strides, multiples of 8 elements (16 bytes) with 16-byte aligned bases; the
 * routes may have any strides (fa4_sparse_gqa_attention accepts noncontiguous
 * IDs).  O, dO, dQ, dK, dV, LSE are dense row-major in the shapes above. */
typedef struct qsa_problem {
    int64_t B, S_q, S_kv, Hq, Hkv, D, K;
    int32_t route_bits;
    float softmax_scale;
    int64_t q_stride[4];
    int64_t k_stride[4];
    int64_t v_stride[4];
    int64_t r_stride[3];
    uint32_t flags; /* 0, or QSA_ROUTES_SORTED | QSA_DETERMINISTIC_FORWARD */
} qsa_problem;

/* qsa_problem.flags: every row's valid IDs are strictly ascending and come before its invalid slots (as
 * qsa_select_token_ids writes its rows).  qsa_preprocess then checks that on each row and copies such rows
 * through instead of sorting them; a row found unsorted is sorted as usual, so the flag never changes a
 * result, only the time (without it, the check is skipped: it would slow unsorted rows down). */
#define QSA_ROUTES_SORTED 1u
/* qsa_problem.flags: qsa_forward's O and LSE bitwise reproducible.  The key-major forward sums each row's
 * output over work items in fp32 in whatever order the items finish, so repeated calls agree within
 * rounding only; with this flag the preprocessing always picks the tile forward (every output row computed
 * by one CTA in a fixed order), slower on routes that a query tile shares poorly.  Together with
 * qsa_backward_deterministic the whole step is reproducible. */
#define QSA_DETERMINISTIC_FORWARD 2u

/* Validates a problem without touching the device. */
QSA_API qsa_status qsa_check_problem(const qsa_problem *problem);

/* Bytes of device workspace qsa_preprocess/qsa_forward/qsa_backward need for
 * this problem (256-byte aligned base required), or 0 if the problem is
 * invalid.  The workspace holds the preprocessed routes (per-row sorted unique
 * IDs and counts; per-query-tile key lists and membership masks; per 64-key
 * chunk, the lists of query rows that route into it, cut into work items),
 * the forward's row statistics and the fp32 accumulator shared by the
 * key-major forward's O and the backward's dQ, the backward's fp32 row
 * statistics and dK/dV accumulators, the work queue counters of the attention
 * kernels, and a device status word.  qsa_preprocess and qsa_forward use only
 * a leading part of the layout and accept a workspace of that size; the
 * backward needs all of it.  Every call that takes the workspace updates it,
 * so calls sharing one workspace must be ordered (one stream, or events
 * between streams). */
QSA_API size_t qsa_workspace_bytes(const qsa_problem *problem);

/* Route preprocessing (fa4_qsa _preprocess and _block_kinds/_compact_blocks
 * play this role on the pages): validates every route ID against [0, S_kv) in
 * its own width before any narrowing, drops duplicates, sorts each row
 * ascending (rows already sorted are copied through when problem->flags has
 * QSA_ROUTES_SORTED), and builds what the attention kernels read: for each
 * aligned 64-key chunk, the query rows that route into it with their key masks
 * (the key-major kernels' work), and, when a tile kernel will run, per query
 * tile the union of its rows' keys with membership masks.  It also decides on
 * the device, from counts of both, which kernel family the forward and the
 * backward use (they compute the same function).  Writes only into
 * `workspace`, which the forward and backward calls then read; reuse it for
 * both as long as the routes are unchanged.  No host synchronisation. */
QSA_API qsa_status qsa_preprocess(const qsa_problem *problem, const void *routes, void *workspace, size_t ws_bytes,
                          cudaStream_t stream);

/* Forward pass (flex_sparse_gqa_attention / fa4_sparse_gqa_attention returns O;
 * the per-row LSE is kept for the backward pass).  Needs a workspace filled by
 * qsa_preprocess for the same problem; the preprocessed routes are only read,
 * the work queue counters are used and left reset.  The key-major forward
 * accumulates O in fp32 through L2 and normalises once at the end; its
 * exponent reference per row is a Cauchy-Schwarz bound on the row's scores
 * when that keeps the row's largest weight above 2^-64, else the row maximum
 * from an extra pass (the same function either way, up to rounding).  o and lse are written in
 * full (rows with no valid route get O = 0 and LSE = -inf); they must not
 * overlap q, k, v or the workspace. */
QSA_API qsa_status qsa_forward(const qsa_problem *problem, void *workspace, size_t ws_bytes, const void *q,
                       const void *k, const void *v, void *o, float *lse, cudaStream_t stream);

/* First-order backward (fa4_sparse_gqa_attention: first-order autograd only,
 * nondeterministic accumulation accepted).  Given O and LSE from qsa_forward and
 * dout = dL/dO, writes dq [B,S_q,Hq,D], dk and dv [B,S_kv,Hkv,D] in BF16.  The
 * sums run in fp32, partly by scatter-add in an order that varies between calls
 * (dQ too on the key-major path), so repeated calls agree within rounding, not
 * bit for bit (qsa_backward_deterministic does); when dk_f32/dv_f32 are non-null they
 * receive those fp32 sums (same shape, float32) and serve as the accumulators,
 * otherwise the workspace does.  Rows with no valid route give dq = 0 and add
 * nothing to dk/dv.  Outputs must not overlap the inputs or each other. */
QSA_API qsa_status qsa_backward(const qsa_problem *problem, void *workspace, size_t ws_bytes, const void *q, const void *k,
                        const void *v, const void *o, const float *lse, const void *dout, void *dq, void *dk,
                        void *dv, float *dk_f32, float *dv_f32, cudaStream_t stream);

/* The same backward with bitwise reproducible dK/dV (and dQ): no counterpart on
 * the pages, whose FA4 backward has no deterministic mode (fa4_qsa
 * fa4_sparse_gqa_attention).  Every dK/dV contribution x is rounded once to the
 * integer round(x * 2^24); the GPU sums those integers modulo 2^32 (integer
 * addition: exact in any order) next to an ordinary fp32 sum of x, and the exact
 * sum is recovered as the value congruent to the integer sum modulo 2^32 that
 * is nearest to the fp32 estimate (which stays far closer than the 2^7 that
 * requires).  The results depend on the inputs only; they are converted to fp32
 * (dk_f32/dv_f32 when non-null) and BF16.  Resolution 2^-24 per contribution.
 * dQ is summed the same way where it is scattered (key-major path) and in a
 * fixed order otherwise.  Costs one more 32-bit reduction per contribution
 * than qsa_backward.  Arguments, layouts and errors
 * are those of qsa_backward; the accumulators live in the workspace. */
QSA_API qsa_status qsa_backward_deterministic(const qsa_problem *problem, void *workspace, size_t ws_bytes,
                                              const void *q, const void *k, const void *v, const void *o,
                                              const float *lse, const void *dout, void *dq, void *dk, void *dv,
                                              float *dk_f32, float *dv_f32, cudaStream_t stream);

/* Copies the preprocessed routes out of the workspace (device to device, on
 * `stream`): ids [B,S_q,K] int32 = each row's valid IDs ascending and
 * deduplicated, then -1; counts [B,S_q] int32 = how many.  Either output may be
 * null.  For bit-exact checks and for counting useful work. */
QSA_API qsa_status qsa_copy_route_sets(const qsa_problem *problem, const void *workspace, size_t ws_bytes, int32_t *ids,
                               int32_t *counts, cudaStream_t stream);

/* Route preprocessing and forward pass in one call that allocates nothing and
 * takes no workspace; the pages have no counterpart to it.  It is meant for
 * callers that cannot allocate device memory while they run (code executing
 * inside a framework that owns all device memory, such as an inference engine
 * plugin's enqueue, or a latency-critical loop that cannot afford an
 * allocation's implicit synchronisation).  Instead of a caller workspace it
 * uses one fixed 32 MiB device array inside the library, which every GPU that
 * loads it keeps until the process exits; problems whose preprocessing and
 * forward regions of the workspace exceed 32 MiB are rejected with
 * QSA_ERR_UNSUPPORTED.  The first call on a device looks up that array's
 * device address (with the device current) and keeps it, so make that first
 * call before any stream capture, and make no further call after
 * cudaDeviceReset on that device.  All calls share the one array and it keeps
 * the last call's contents: calls that overlap on the GPU (other streams,
 * other host threads) race with each other.  Outputs and conventions are
 * those of qsa_preprocess + qsa_forward; device-side failures are read with
 * qsa_read_no_alloc_status. */
QSA_API qsa_status qsa_forward_no_alloc(const qsa_problem *problem, const void *routes, const void *q, const void *k,
                                        const void *v, void *o, float *lse, cudaStream_t stream);

/* Synchronises `stream`, then reads and clears the device status word of
 * qsa_forward_no_alloc's array on the current device (what
 * qsa_read_device_status does for a caller workspace).  Blocks the host. */
QSA_API qsa_status qsa_read_no_alloc_status(cudaStream_t stream);

/* Synchronises `stream`, then reads and clears the workspace's device status
 * word: QSA_ERR_TIMEOUT if a kernel's bounded wait gave up, QSA_ERR_DEVICE_CHECK
 * if a device bounds check fired, QSA_OK otherwise.  Blocks the host. */
QSA_API qsa_status qsa_read_device_status(const void *workspace, cudaStream_t stream);

/* Static description of a status code. */
QSA_API const char *qsa_status_string(qsa_status status);

/* One-line reason for the last error returned on this host thread ("" if none). */
QSA_API const char *qsa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H_ */
