// Internal launcher of the activation quantization kernel (used by the GEMV
// and MoE entry points to chain it in front of their own kernel).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace rfp2 {

// One warp quantizes 32-value block b of x, one lane per value: d = max|a| /
// 127 and q = round-half-away(a / d) (0 when d == 0), both divisions IEEE
// round-to-nearest, so the codes match the oracle bit for bit.
RFP2_DEV void quantize_block_warp(const float *__restrict__ x, int64_t b, int lane,
                                  int8_t *__restrict__ q, float *__restrict__ d) {
    const float a = x[b * 32 + lane];
    float amax = fabsf(a);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float dd = __fdiv_rn(amax, 127.0f);
    int v = 0;
    if (dd != 0.0f) {
        float r = roundf(__fdiv_rn(a, dd));
        r = fminf(fmaxf(r, -127.0f), 127.0f);
        v = static_cast<int>(r);
    }
    q[b * 32 + lane] = static_cast<int8_t>(v);
    if (lane == 0) d[b] = dd;
}

// Enqueue the quantization of x [N, K] into q [N, K] and d [N, K/32].  With
// pdl = true the kernel is launched with programmatic stream serialization:
// it waits for the previous kernel itself and lets the next one start early.
cudaError_t launch_quantize(const float *x, int64_t N, int64_t K, int8_t *q, float *d,
                            cudaStream_t stream, bool pdl);

}  // namespace rfp2
