// qsa_tc_host.cu -- host helpers of the tile kernels: TMA tensor-map encoding
// (through the driver entry point, so the library does not link libcuda) and
// device capability checks.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <mutex>

#include "qsa_tc.cuh"

namespace qsa {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

}  // namespace

bool tc_device_ok() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return false;
    return major == 10 && minor == 3 && encode_fn() != nullptr;
}

int tc_num_sms() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

uint64_t tc_wait_limit_ns(uint64_t fallback) {
    const char *env = std::getenv("QSA_DEBUG_WAIT_LIMIT_NS");
    if (!env || !*env) return fallback;
    char *end = nullptr;
    const unsigned long long v = std::strtoull(env, &end, 10);
    return (end && *end == '\0') ? (uint64_t)v : fallback;
}

bool tc_encode_rows_map(CUtensorMap *m, const void *base, int64_t rows, int64_t row_stride_elems, int64_t D) {
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_stride_elems * 2};
    const cuuint32_t box[2] = {64, 1};
    const cuuint32_t estr[2] = {1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_encode_run_map(CUtensorMap *m, const void *base, int64_t rows, int64_t row_stride_elems, int64_t D) {
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_stride_elems * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kChunkKeys};
    const cuuint32_t estr[2] = {1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_encode_kv_maps(KVMaps *m, const AttnArgs &a, int64_t b, int64_t g) {
    const __nv_bfloat16 *kb = a.k + b * a.ks0 + g * a.ks2, *vb = a.v + b * a.vs0 + g * a.vs2;
    return tc_encode_rows_map(&m->k_rows, kb, a.S_kv, a.ks1, a.D) &&
           tc_encode_rows_map(&m->v_rows, vb, a.S_kv, a.vs1, a.D) && tc_encode_run_map(&m->k_run, kb, a.S_kv, a.ks1, a.D) &&
           tc_encode_run_map(&m->v_run, vb, a.S_kv, a.vs1, a.D);
}

bool tc_encode_tile_map(CUtensorMap *m, const void *base, int64_t H, int64_t S, int64_t B, int64_t sH, int64_t sS,
                        int64_t sB, int64_t G, int64_t T, int64_t D) {
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)sH * 2, (cuuint64_t)sS * 2, (cuuint64_t)sB * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)T, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_head_major_order(const AttnArgs &a, int64_t n_g) {
    int dev = 0, bytes = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&bytes, cudaDevAttrL2CacheSize, dev);
    const int64_t l2 = bytes > 0 ? bytes : (64ll << 20);
    const int64_t acc_bytes = a.B * a.S_kv * n_g * a.D * 2 * (int64_t)sizeof(float);
    return acc_bytes > l2 / 2;
}

bool tc_encode_bf16_map(CUtensorMap *m, const void *base, int rank, const int64_t *dims, const int64_t *strides,
                        const uint32_t *box) {
    if (rank < 2 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t bx[5], estr[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = (cuuint64_t)dims[i];
        bx[i] = box[i];
        estr[i] = 1;
        if (i > 0) st[i - 1] = (cuuint64_t)strides[i - 1] * 2;
    }
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base), d, st, bx, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace qsa
