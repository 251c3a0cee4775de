// qsa_tc.cuh -- tile (tensor-core) path of libqsa: shared declarations.
#pragma once

#include <cuda.h>

#include "qsa_internal.cuh"

namespace qsa {

// Per-tile preprocessed routes in the workspace (see qsa_preprocess.cu).
struct TileArgs {
    int64_t T;           // queries per tile (kTileRows / G)
    int64_t n_tiles;     // tiles per batch row
    int64_t max_chunks;  // chunk capacity of one tile
    const int32_t *tile_nchunks;
    const int32_t *tile_keys;
    const uint64_t *tile_masks;
    const int32_t *order;
    int32_t *sched;  // {next, done} work queue counters: [0..1] forward, [2..3] backward; zero between launches
};

// Host helpers shared by the tile kernels (qsa_tc_host.cu).
bool tc_device_ok();  // current device is sm_103 and the TMA map encoder is reachable
int tc_num_sms();
// Bound of the tile kernels' pipeline waits: `fallback` unless the environment
// variable QSA_DEBUG_WAIT_LIMIT_NS sets it (a test hook that makes a wait run
// out on purpose; the kernels then report QSA_ERR_TIMEOUT and wind down).
uint64_t tc_wait_limit_ns(uint64_t fallback);
// 2-D map over `rows` rows of D bf16 (row pitch in elements), box 64 x 1,
// 128-byte swizzle: the operand of tile::gather4 row gathers.
bool tc_encode_rows_map(CUtensorMap *m, const void *base, int64_t rows, int64_t row_stride_elems,
                        int64_t D = kHeadDim);
// Same tensor with a 64 x 64 box: one tile load brings 64 consecutive rows
// (a contiguous run of keys) in the layout the 64-row gathers produce.
bool tc_encode_run_map(CUtensorMap *m, const void *base, int64_t rows, int64_t row_stride_elems,
                       int64_t D = kHeadDim);

// Tensor maps of one (batch, KV head) pair: K and V for row gathers and for
// 64-row contiguous runs.
struct KVMaps {
    CUtensorMap k_rows, v_rows, k_run, v_run;
};
constexpr int kMaxKVPairs = 32;  // pairs per launch (kernel parameter space)
bool tc_encode_kv_maps(KVMaps *m, const AttnArgs &a, int64_t b, int64_t g);
// 4-D map over a [B, S, H, D] bf16 tensor (strides in elements), box
// {64, G, T, 1}, 128-byte swizzle: one (T queries x G heads) tile per 64 columns.
bool tc_encode_tile_map(CUtensorMap *m, const void *base, int64_t H, int64_t S, int64_t B, int64_t sH, int64_t sS,
                        int64_t sB, int64_t G, int64_t T, int64_t D = kHeadDim);

// Generic BF16 tensor map, 128-byte swizzle, zero fill out of bounds: dims[0]
// is the innermost (unit-stride) extent, strides[i] (elements) the pitch of
// dimension i + 1, box the tile extents.
bool tc_encode_bf16_map(CUtensorMap *m, const void *base, int rank, const int64_t *dims, const int64_t *strides,
                        const uint32_t *box);

// Work queue order of a tile-kernel launch over n_g KV heads: head by head when
// those heads' fp32 dK/dV accumulators together exceed half of L2 (the K/V
// rows and Q/dO tiles share the rest), else interleaved.
bool tc_head_major_order(const AttnArgs &a, int64_t n_g);

bool tc_forward_supported();
bool tc_forward_shape_ok(const AttnArgs &a, const TileArgs &t);
// choice: null, or a device flag; the tile forward returns at once when *choice == 1 (the key-major
// forward runs instead).
cudaError_t launch_tc_forward(const AttnArgs &a, const TileArgs &t, __nv_bfloat16 *o, float *lse,
                              const int32_t *choice, cudaStream_t s);

// Key-major backward (qsa_bwd_km.cu): reverse lists from qsa_chunks.cu and the
// fp32 dQ accumulator it scatter-adds into.
struct KmArgs {
    int64_t NC;  // aligned 64-key chunks per batch row
    const int4 *items;
    const int32_t *queue, *meta, *e_q;
    const uint64_t *e_mask;
    int32_t *sched;  // work queue counters {next, done}
    float *dq_acc;   // fp32 [B, S_q, Hq, D] (zeroed), or null in deterministic mode
    FxAcc dq_fx;     // deterministic mode: exact accumulators
    const int32_t *gate;  // null, or a device flag: the kernel and its dQ conversion run only when *gate == 1
};
bool km_backward_shape_ok(const AttnArgs &a);
cudaError_t launch_km_backward(const BwdArgs &b, const KmArgs &k, cudaStream_t s);

// Key-major forward (qsa_fwd_km.cu): the same reverse lists and work queue, two passes (row maxima, then
// outputs reduced into fp32 accumulators) and a final division.  launch_km_choose decides on the device,
// from the preprocessed routes, whether it or the tile forward runs: choice[0] = 1 for the key-major one.
struct KfArgs {
    int64_t NC;
    const int4 *items;
    const int32_t *queue, *meta, *e_q;
    const uint64_t *e_mask;
    int32_t *sched;   // two pairs of work queue counters {next, done}: row-max pass, output pass
    int32_t *mrow;    // [B, S_q, Hq] encoded row maxima
    float *mref;      // [B, S_q, Hq] exponent references from the norm bound
    float *lrow;      // [B, S_q, Hq] pairs: sums of P and of P rounded to BF16
    float *o_acc;     // [B, S_q, Hq, D] fp32
    const int32_t *choice;
    int32_t *kbound;  // [kKeyNormWord + B * Hkv]: {row-max pass needed, ...}, then squared key norm maxima
};
constexpr int64_t kKeyNormWord = 64;
bool km_forward_shape_ok(const AttnArgs &a);
int forced_path(const char *env_var);  // debug override of a path choice: 0 tile, 1 key-major, -1 none
// choice[0]: 1 = key-major forward (never with tile_fwd_only); choice[1]: 1 = key-major backward (always 1
// when !tile_bwd_ok).
cudaError_t launch_km_choose(const int32_t *tile_keys, int64_t n_tiles, const int32_t *list_start,
                             int64_t n_lists, int64_t slots, int64_t D, bool tile_bwd_ok, bool tile_fwd_only,
                             int32_t *choice, cudaStream_t s);
cudaError_t launch_km_forward(const AttnArgs &a, const KfArgs &k, __nv_bfloat16 *o, float *lse, cudaStream_t s);

bool tc_backward_supported();
bool tc_backward_shape_ok(const AttnArgs &a, const TileArgs &t);
// gate: null, or a device flag; the tile backward returns at once when *gate == 1 (the key-major one runs).
cudaError_t launch_tc_backward(const BwdArgs &b, const TileArgs &t, const int32_t *gate, cudaStream_t s);

}  // namespace qsa
