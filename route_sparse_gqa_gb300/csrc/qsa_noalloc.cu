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
// per device (with that device current) on the first call made there.
#include <mutex>

#include "qsa_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 128;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices];

}  // namespace

extern "C" QSA_API qsa_status qsa_forward_no_alloc(const qsa_problem *problem, const void *routes, const void *q,
                                                   const void *k, const void *v, void *o, float *lse,
                                                   cudaStream_t stream) {
    qsa_status st = qsa_check_problem(problem);
    if (st != QSA_OK) return st;
    const size_t need = qsa_workspace_bytes(problem);
    if (need > kNoAllocScratchBytes)
        return qsa::report_error(QSA_ERR_UNSUPPORTED,
                                 "problem too large for qsa_forward_no_alloc: its workspace exceeds the fixed 32 MiB "
                                 "device scratch; use qsa_preprocess + qsa_forward with a caller workspace");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return qsa::report_error(QSA_ERR_CUDA, "qsa_forward_no_alloc: no usable current device");
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_scratch_addr[dev]) {
            void *addr = nullptr;
            e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
            if (e != cudaSuccess || !addr)
                return qsa::report_error(QSA_ERR_CUDA, "qsa_forward_no_alloc: cudaGetSymbolAddress failed");
            g_scratch_addr[dev] = addr;
        }
        scratch = g_scratch_addr[dev];
    }
    // qsa_preprocess clears the status word and rewrites every scratch region
    // the forward kernel reads, so nothing left by an earlier call leaks in.
    st = qsa_preprocess(problem, routes, scratch, kNoAllocScratchBytes, stream);
    if (st != QSA_OK) return st;
    return qsa_forward(problem, scratch, kNoAllocScratchBytes, q, k, v, o, lse, stream);
}
