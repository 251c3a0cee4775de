// qsa_tc.cuh -- tile (tensor-core) path of libqsa: shared declarations.
#pragma once

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
};

bool tc_forward_supported();
bool tc_forward_shape_ok(const AttnArgs &a, const TileArgs &t);
cudaError_t launch_tc_forward(const AttnArgs &a, const TileArgs &t, __nv_bfloat16 *o, float *lse, cudaStream_t s);

bool tc_backward_supported();
cudaError_t launch_tc_backward(const BwdArgs &b, const TileArgs &t, cudaStream_t s);

}  // namespace qsa
