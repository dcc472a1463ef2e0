// Q8_1-style activation quantization: fp32 [N, K] -> int8 [N, K] + fp32
// d [N, K/32], d = max|a| / 127, q = round-half-away(a / d), q = 0 when d == 0.
//
// Source: "ROCmFP2 codebook research report", section "03 Runtime" (the
// weights are dotted against Q8_1 activations; the per-32 scale d = max|a|/127
// in fp32 is the statement of the problem).  One warp per 32-value block, one
// lane per value: the absolute maximum is a warp reduction (exact, so its
// order does not matter), both divisions are IEEE round-to-nearest so the
// int8 codes match the oracle bit for bit.
#include "common.cuh"
#include "quantize.cuh"

namespace rfp2 {

__global__ void __launch_bounds__(256) quantize_act_kernel(const float *__restrict__ x,
                                                           int64_t nblocks,
                                                           int8_t *__restrict__ q,
                                                           float *__restrict__ d) {
    // When chained after another kernel with programmatic dependent launch,
    // wait for it, then let the consumer of q/d start its own prologue.
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t b = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < nblocks;
         b += warps)
        quantize_block_warp(x, b, lane, q, d);
}

cudaError_t launch_quantize(const float *x, int64_t N, int64_t K, int8_t *q, float *d,
                            cudaStream_t stream, bool pdl) {
    const int64_t nblocks = N * (K / 32);
    if (nblocks == 0) return cudaSuccess;
    const int warps_per_cta = 8;
    int64_t ctas = (nblocks + warps_per_cta - 1) / warps_per_cta;
    const int64_t cap = 8LL * sm_count(current_device());
    if (ctas > cap) ctas = cap;
    return launch(quantize_act_kernel, dim3((unsigned)ctas), dim3(warps_per_cta * 32), 0, stream,
                  pdl, x, nblocks, q, d);
}

}  // namespace rfp2

extern "C" rfp2_status rfp2_quantize_act(const float *x, int64_t N, int64_t K, int8_t *q,
                                         float *d, rfp2_stream_t stream) {
    if (N < 0 || K < 0) return RFP2_EINVAL;
    if (K % 32 != 0) return RFP2_ESHAPE;
    if (N == 0 || K == 0) return RFP2_OK;
    if (!x || !q || !d) return RFP2_EINVAL;
    if (!rfp2::aligned(x, 4) || !rfp2::aligned(d, 4)) return RFP2_EALIGN;
    return rfp2::from_cuda(
        rfp2::launch_quantize(x, N, K, q, d, reinterpret_cast<cudaStream_t>(stream), false));
}
