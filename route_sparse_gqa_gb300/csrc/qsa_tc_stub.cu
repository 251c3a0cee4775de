// qsa_tc_stub.cu -- placeholder until the tensor-core kernels land.
#include "qsa_tc.cuh"

namespace qsa {
bool tc_forward_supported() { return false; }
cudaError_t launch_tc_forward(const AttnArgs &, const TileArgs &, __nv_bfloat16 *, float *, cudaStream_t) {
    return cudaErrorNotSupported;
}
bool tc_backward_supported() { return false; }
cudaError_t launch_tc_backward(const BwdArgs &, const TileArgs &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace qsa
