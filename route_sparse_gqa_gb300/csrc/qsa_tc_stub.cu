// qsa_tc_stub.cu -- placeholder until the tensor-core kernels land.
#include "qsa_tc.cuh"

namespace qsa {
bool tc_backward_supported() { return false; }
cudaError_t launch_tc_backward(const BwdArgs &, const TileArgs &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace qsa
