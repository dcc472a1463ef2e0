// ABI bookkeeping of librfp2: status strings, version, per-device SM counts.
#include <mutex>

#include "common.cuh"

namespace rfp2 {

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

}  // namespace rfp2

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
