// qsa_internal.cuh -- shared definitions of the libqsa CUDA sources (not installed).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qsa.h"

namespace qsa {

constexpr int kHeadDim = 256;        // fa4_sparse_gqa_attention fixes D = 256 (the tile kernels' head dim)
constexpr int kChunkKeys = 64;       // keys per gathered chunk (one tensor-core N tile)
constexpr int kTileRows = 128;       // (query, head) rows per tile = tcgen05 M
constexpr int kMaxRouteSlots = 16384;  // per-row sort capacity (smem bitonic sort)

// Device status word kept at the start of the workspace.  Kernels only ever
// raise it (atomicCAS from 0); qsa_read_device_status reads and clears it.
struct DeviceStatus {
    unsigned int code;       // 0 = ok, else a qsa_status value
    unsigned int where;      // kernel-specific site id of the first failure
    unsigned int info0, info1;
};

// Workspace layout for one problem.  All offsets are 256-byte aligned.
struct Layout {
    int64_t G;           // query heads per KV head
    int64_t T;           // queries per tile (kTileRows / G), 0 when the tile path does not apply
    int64_t n_tiles;     // query tiles per batch row
    int64_t max_chunks;  // capacity of one tile's chunk list
    size_t off_status, off_sched, off_counts, off_ids, off_tile_nchunks, off_tile_keys, off_tile_masks, off_order;
    size_t fwd_total;  // bytes the preprocessing and the forward use (everything before the backward's regions)
    // Key-major paths (qsa_chunks.cu, qsa_fwd_km.cu, qsa_bwd_km.cu); km = false when the problem does not take them.
    bool km;
    int64_t NC, n_blk_b, win_blocks, n_win_b, max_groups, cap_entries, cap_items;
    size_t off_rmask, off_hoff, off_list_start, off_eq, off_emask, off_part_start, off_items, off_sorted, off_queue, off_kmeta,
        off_tkeys;
    size_t off_mrow, off_mref, off_lrow, off_kbound;  // key-major forward row statistics and key norm bound
    size_t off_delta, off_dk, off_dv, off_dq, total;  // off_dk/off_dv/off_dq: 8 bytes per element (fp32 or fixed point)
};

// Workspace bytes the preprocessing and the forward need (a prefix of the full layout).
size_t forward_workspace_bytes(const qsa_problem *p);

// Device-side failure sites (DeviceStatus::where).
enum Site : unsigned int {
    kSiteNone = 0,
    kSiteRowwiseFwdId = 1,
    kSiteRowwiseBwdId = 2,
    kSiteTileFwdWait = 10,
    kSiteTileFwdKey = 11,
    kSiteTileBwdWait = 20,
    kSiteTileBwdKey = 21,
    kSiteKeyBwdWait = 22,
    kSiteKeyFwdWait = 23,
    kSiteChunkCapacity = 24,
    kSiteRouteScoreWait = 30,
};

__device__ __forceinline__ void raise_status(DeviceStatus *st, unsigned int code, unsigned int where,
                                             unsigned int i0 = 0, unsigned int i1 = 0) {
    if (atomicCAS(&st->code, 0u, code) == 0u) {
        st->where = where;
        st->info0 = i0;
        st->info1 = i1;
    }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float f[8]) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 f32x8_to_bf16(const float f[8]) {
    uint4 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return u;
}

// Records `msg` as the calling thread's qsa_last_error() and returns `st`.
qsa_status report_error(qsa_status st, const char *msg);

// ---- launch wrappers implemented in the .cu files (return cudaGetLastError()) ----

struct RowsArgs {
    const void *routes;
    int32_t route_bits;
    int64_t B, S_q, S_kv, K;
    int64_t rs0, rs1, rs2;
    int32_t *ids;     // [B*S_q, K]
    int32_t *counts;  // [B*S_q]
    bool try_sorted;  // QSA_ROUTES_SORTED: copy rows found sorted through
};
cudaError_t launch_route_rows(const RowsArgs &a, cudaStream_t s);

struct TilesArgs {
    int64_t B, S_q, S_kv, K, T, n_tiles, max_chunks, Hkv;
    const int32_t *ids;
    const int32_t *counts;
    int32_t *tile_nchunks;    // [B*n_tiles]
    int32_t *tile_keys;       // [B*n_tiles, max_chunks*64]
    uint64_t *tile_masks;     // [B*n_tiles, max_chunks, T]
    int32_t *order;           // [B*n_tiles*Hkv] work items, heaviest first
    const int32_t *skip;      // if set and skip[0] == skip[1] == 1 (key-major forward and backward), nothing is built
};
cudaError_t launch_route_tiles(const TilesArgs &a, cudaStream_t s);

// Key-major (reverse-route) lists, built from the sorted route sets for the
// key-major backward (qsa_chunks.cu).  Key space is cut into aligned chunks of
// 64 keys, NC per batch row; list (b, c) holds one entry per query row of
// batch b that routes into chunk c: the query index and the 64-bit mask of the
// chunk keys it routes to, in ascending query order.  Query rows are taken in
// blocks of 64; a list is cut into parts (work items) of at most max_groups
// groups of `slots` entries whose queries lie in one window of win_blocks
// blocks; the work queue runs window by window, KV head by KV head within a
// window, largest parts first.
struct ChunkArgs {
    int64_t B, S_q, S_kv, K, NC, Hkv;
    int64_t n_blk_b;     // 64-row query blocks per batch row
    int64_t win_blocks;  // blocks per window
    int64_t n_win_b;     // windows per batch row
    int64_t slots;       // queries per group (one MMA tile: 128 / G)
    int64_t max_groups;  // groups per part at most
    int64_t cap_entries, cap_items;
    const int32_t *ids, *counts;
    uint64_t *rmask;      // [B * n_blk_b, NC]: which of the block's 64 rows route into each chunk
    int32_t *hoff;        // [B * n_blk_b, NC]: where the block's entries start inside each list
    int32_t *list_start;  // [B * NC + 1]: exclusive scan of list lengths
    int32_t *e_q;         // [cap_entries]: query index of each entry
    uint64_t *e_mask;     // [cap_entries]: chunk keys the query routes to
    int32_t *part_start;  // [B * NC + 1]: parts per list, then their exclusive scan
    int4 *items;          // [cap_items]: {list, first entry, entries, window}
    int32_t *sorted;      // [cap_items]: items by window, largest first
    int32_t *queue;       // [cap_items * Hkv]: item * Hkv + KV head, in work order
    int32_t *meta;        // {entries, items, queue length, overflow flag}
    int32_t *tile_keys;   // [B * ceil(S_q / slots)]: distinct routed keys of each query tile (null: not needed)
    DeviceStatus *status;  // raised (QSA_ERR_DEVICE_CHECK) if a capacity would be exceeded
};
cudaError_t launch_chunk_lists(const ChunkArgs &a, cudaStream_t s);

struct AttnArgs {
    int64_t B, S_q, S_kv, Hq, Hkv, K, G;
    int64_t D;  // head dim: 256 on the tile path; 64, 128 or 256 on the warp-level path
    float scale;
    const __nv_bfloat16 *q, *k, *v;
    int64_t qs0, qs1, qs2, ks0, ks1, ks2, vs0, vs1, vs2;
    const int32_t *ids, *counts;
    DeviceStatus *status;
};

cudaError_t launch_rowwise_forward(const AttnArgs &a, __nv_bfloat16 *o, float *lse, cudaStream_t s);

// Deterministic dK/dV.  Every contribution x is rounded once to the integer
// c = round(x * 2^24).  Two 32-bit reductions per element: `lo` sums c modulo
// 2^32 (integer addition: exact and independent of order) and `est` sums x in
// fp32 (order-dependent rounding, but within far less than 2^31 / 2^24 = 128 of
// the exact sum).  The exact integer sum is the one value congruent to `lo`
// modulo 2^32 nearest to est * 2^24, so the result depends on the inputs only:
// bitwise reproducible.  Resolution 2^-24 per contribution.
struct FxAcc {
    float *est;    // [n] fp32 running sums
    uint32_t *lo;  // [n] sums of round(x * 2^24) modulo 2^32
};

constexpr float kFxScale = 16777216.0f;  // 2^24

__device__ __forceinline__ void red_add_fx(float *est, uint32_t *lo, float x) {
    const uint32_t c = (uint32_t)(unsigned long long)__float2ll_rn(x * kFxScale);
    asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(est), "f"(x) : "memory");
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(lo), "r"(c) : "memory");
}

__device__ __forceinline__ void red_add_fx(const FxAcc &acc, int64_t i, float x) { red_add_fx(acc.est + i, acc.lo + i, x); }

__device__ __forceinline__ float fx_to_f32(float est, uint32_t lo) {
    const double e = (double)est * (double)kFxScale;
    const long long k = __double2ll_rn((e - (double)lo) * (1.0 / 4294967296.0));
    const long long sum = (long long)lo + k * 4294967296ll;
    return (float)((double)sum * (1.0 / (double)kFxScale));
}

struct BwdArgs {
    AttnArgs f;
    const __nv_bfloat16 *o, *dout;
    const float *lse;
    float *delta;  // [B, Hq, S_q]
    __nv_bfloat16 *dq, *dk, *dv;
    float *dk_acc, *dv_acc;  // fp32 [B, S_kv, Hkv, D]: the accumulators, or (deterministic) fp32 outputs / null
    // Deterministic mode: exact accumulators (see FxAcc), else est = null.
    FxAcc dk_fx, dv_fx;
};

cudaError_t launch_rowwise_backward(const BwdArgs &a, cudaStream_t s);  // deterministic when a.dk_fx.est is set
cudaError_t launch_delta(const BwdArgs &a, cudaStream_t s);
cudaError_t launch_convert_dkdv(const BwdArgs &a, cudaStream_t s);  // from a.dk_fx when a.dk_fx.est is set

}  // namespace qsa
