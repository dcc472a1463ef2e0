// Internal launcher of the activation quantization kernel (used by the GEMV
// and MoE entry points to chain it in front of their own kernel).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rfp2 {

// Enqueue the quantization of x [N, K] into q [N, K] and d [N, K/32].  With
// pdl = true the kernel is launched with programmatic stream serialization:
// it waits for the previous kernel itself and lets the next one start early.
cudaError_t launch_quantize(const float *x, int64_t N, int64_t K, int8_t *q, float *d,
                            cudaStream_t stream, bool pdl);

}  // namespace rfp2
