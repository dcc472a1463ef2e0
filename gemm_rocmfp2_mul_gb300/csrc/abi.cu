// ABI bookkeeping of librfp2: status strings, version, per-device SM counts,
// the process-wide weight-prefetch switch.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "tma.cuh"

namespace rfp2 {

// cuTensorMapEncodeTiled through the runtime's driver entry point (so the
// library does not link libcuda itself).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool encode_tensor_map_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype,
                          uint64_t cols, uint64_t rows, uint64_t row_bytes, uint32_t box_cols,
                          uint32_t box_rows, CUtensorMapSwizzle swizzle) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t elem_strides[2] = {1, 1};
    const CUresult r = fn(map, dtype, 2, const_cast<void *>(base), dims, strides, box, elem_strides,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_tensor_map_3d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype,
                          const uint64_t (&dims)[3], const uint64_t (&strides)[2],
                          const uint32_t (&box)[3], CUtensorMapSwizzle swizzle) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    cuuint64_t st[2] = {strides[0], strides[1]};
    cuuint32_t b[3] = {box[0], box[1], box[2]};
    cuuint32_t elem_strides[3] = {1, 1, 1};
    const CUresult r = fn(map, dtype, 3, const_cast<void *>(base), d, st, b, elem_strides,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int current_device() {
    int dev = 0;
    cudaGetDevice(&dev);
    return dev;
}

int sm_count(int device) {
    static std::mutex mu;
    static int cache[64] = {0};
    if (device < 0 || device >= 64) device = 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[device] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
            n <= 0)
            n = 1;
        cache[device] = n;
    }
    return cache[device];
}

cudaError_t launch_status() { return cudaGetLastError(); }

// Off by default: every kernel waits for the work enqueued before it on its
// stream before reading weights.
static std::atomic<int> g_weight_prefetch{0};

bool weight_prefetch() { return g_weight_prefetch.load(std::memory_order_relaxed) != 0; }

}  // namespace rfp2

extern "C" rfp2_status rfp2_set_weight_prefetch(int enable) {
    rfp2::g_weight_prefetch.store(enable ? 1 : 0, std::memory_order_relaxed);
    return RFP2_OK;
}

extern "C" int rfp2_weight_prefetch(void) { return rfp2::weight_prefetch() ? 1 : 0; }

extern "C" const char *rfp2_status_str(int status) {
    switch (status) {
        case RFP2_OK: return "RFP2_OK";
        case RFP2_EINVAL: return "RFP2_EINVAL";
        case RFP2_ESHAPE: return "RFP2_ESHAPE";
        case RFP2_EALIGN: return "RFP2_EALIGN";
        case RFP2_EUNSUPPORTED: return "RFP2_EUNSUPPORTED";
        case RFP2_ECUDA: return "RFP2_ECUDA";
        case RFP2_EBADSCALE: return "RFP2_EBADSCALE";
        case RFP2_EBADID: return "RFP2_EBADID";
        case RFP2_ETIMEOUT: return "RFP2_ETIMEOUT";
        case RFP2_EWORKSPACE: return "RFP2_EWORKSPACE";
    }
    return "RFP2_UNKNOWN";
}

extern "C" int rfp2_version(void) { return 100; }
