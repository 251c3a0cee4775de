// qsa_noalloc.cu -- route preprocessing + forward for callers that must not
// allocate device memory.
//
// Some callers cannot call cudaMalloc while they run: code inside a host
// framework that owns every device byte (an inference engine's plugin
// executing inside its enqueue call, a runtime with a fixed memory plan) or a
// latency-critical loop that cannot afford an allocation's implicit device
// synchronisation.  qsa_forward_no_alloc serves them: its only scratch -- the
// preprocessed routes the forward kernel reads -- lives in the fixed-size
// device array below instead of a caller-provided workspace.
//
// The array is a file-scope __device__ variable, so every GPU on which this
// module is loaded keeps its kNoAllocScratchBytes until the process exits.
// In host code `g_noalloc_scratch` names a host-side shadow, not device
// memory; the device address comes from cudaGetSymbolAddress, looked up once
// per device (with that device current) on the first call made there and
// kept until the process exits (cudaDeviceReset ends the module's device
// copy, so no-alloc calls after a reset are not supported).  Device-side
// failures of a call (a bounded wait that ran out, a bounds check) land in the
// status word at the start of the array: qsa_read_no_alloc_status reads and
// clears it.
#include <mutex>

#include "qsa_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 128;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices];

}  // namespace

namespace {

// The scratch array's device address on the current device, looked up the first time a device is used
// (with that device current) and remembered for the life of the process.
qsa_status scratch_address(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return qsa::report_error(QSA_ERR_CUDA, "no-alloc entry point: no usable current device");
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
        if (e != cudaSuccess || !addr)
            return qsa::report_error(QSA_ERR_CUDA, "no-alloc entry point: cudaGetSymbolAddress failed");
        g_scratch_addr[dev] = addr;
    }
    *out = g_scratch_addr[dev];
    return QSA_OK;
}

}  // namespace

extern "C" QSA_API qsa_status qsa_forward_no_alloc(const qsa_problem *problem, const void *routes, const void *q,
                                                   const void *k, const void *v, void *o, float *lse,
                                                   cudaStream_t stream) {
    qsa_status st = qsa_check_problem(problem);
    if (st != QSA_OK) return st;
    // Only the preprocessing's and the forward's regions of the workspace layout are needed.
    const size_t need = qsa::forward_workspace_bytes(problem);
    if (need > kNoAllocScratchBytes)
        return qsa::report_error(QSA_ERR_UNSUPPORTED,
                                 "problem too large for qsa_forward_no_alloc: its forward workspace exceeds the fixed "
                                 "32 MiB device scratch; use qsa_preprocess + qsa_forward with a caller workspace");
    void *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != QSA_OK) return st;
    // qsa_preprocess clears the status word and rewrites every scratch region
    // the forward kernels read, so nothing left by an earlier call leaks in.
    st = qsa_preprocess(problem, routes, scratch, kNoAllocScratchBytes, stream);
    if (st != QSA_OK) return st;
    return qsa_forward(problem, scratch, kNoAllocScratchBytes, q, k, v, o, lse, stream);
}

extern "C" QSA_API qsa_status qsa_read_no_alloc_status(cudaStream_t stream) {
    void *scratch = nullptr;
    const qsa_status st = scratch_address(&scratch);
    if (st != QSA_OK) return st;
    return qsa_read_device_status(scratch, stream);
}
