// Weight preparation on the GPU: ROCmFP2 and HFP4G32 packers, the ROCmFP2
// scale-byte validator and the debug entry that exposes every int32 half sum.
//
// The packers are offline preparation (not on the timed path) but must give
// the same bytes as the CPU oracle, so every floating-point step is an
// explicitly rounded IEEE operation in the oracle's order (no contraction).
//
// Sources: "ROCmFP2 codebook research report", section "02 Quantization"
// (codebook, UE4M3, code choice by sign and |x/s| <= 2.5, lowest squared
// error); "HFP4" (hipfire.dev), sections "Quantization recipe (HFP4G32)",
// "Byte layout - HFP4G32" and "Nibble packing".
#include <cuda_fp16.h>

#include "common.cuh"
#include "rfp2_decode.cuh"

namespace rfp2 {
namespace {

// UE4M3 byte -> scale, for the packer (same closed form as decode_scale_pair).
__device__ __forceinline__ float ue4m3_scale(int b) {
    return __int_as_float((uint32_t)b << 20) * kTwoPow119;
}

// Level index of x at scale s: 0 -> -4, 1 -> -1, 2 -> +1, 3 -> +4.
__device__ __forceinline__ int code_of(float x, float s) {
    const bool neg = x < 0.0f;
    bool inner = true;
    if (s != 0.0f) inner = fabsf(__fdiv_rn(x, s)) <= 2.5f;
    return neg ? (inner ? 1 : 0) : (inner ? 2 : 3);
}

__device__ __forceinline__ float level_of(int code) {
    return code == 0 ? -4.0f : code == 1 ? -1.0f : code == 2 ? 1.0f : 4.0f;
}

// One thread per 16-value half: exhaustive search over bytes 0x00..0x7E.
__global__ void __launch_bounds__(256) rfp2_pack_kernel(const float *__restrict__ W,
                                                        int64_t nhalves,
                                                        uint8_t *__restrict__ out) {
    const int64_t h = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= nhalves) return;
    float x[16];
    const float4 *src = reinterpret_cast<const float4 *>(W + h * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 t = src[i];
        x[4 * i] = t.x;
        x[4 * i + 1] = t.y;
        x[4 * i + 2] = t.z;
        x[4 * i + 3] = t.w;
    }
    int best = 0;
    double best_sse = 0.0;
    for (int b = 0; b <= 0x7E; ++b) {
        const float s = ue4m3_scale(b);
        double sse = 0.0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float r = __fmul_rn(level_of(code_of(x[i], s)), s);
            const double e = __dsub_rn((double)x[i], (double)r);
            sse = __dadd_rn(sse, __dmul_rn(e, e));
        }
        if (b == 0 || sse < best_sse) {
            best_sse = sse;
            best = b;
        }
    }
    const float s = ue4m3_scale(best);
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) word |= (uint32_t)code_of(x[i], s) << (2 * i);
    const int64_t blk = h >> 1, half = h & 1;
    uint8_t *o = out + blk * 10;
#pragma unroll
    for (int i = 0; i < 4; ++i) o[4 * half + i] = (uint8_t)(word >> (8 * i));
    o[8 + half] = (uint8_t)best;
}

// Importance-weighted scale search ("ROCmFP2 codebook research report",
// section "05 Completed experiment"): every term of the squared error is
// weighted by importance_k * sqrt(sigma^2 + x_k^2), sigma^2 = twice the mean
// of x^2 over the 32-weight block (the page leaves sigma^2 undefined); the
// same IEEE fp64 steps in the same order as the plain search, one thread per
// half.  The block, the codebook and the code rule are unchanged.
__global__ void __launch_bounds__(256) rfp2_pack_weighted_kernel(const float *__restrict__ W,
                                                                 const float *__restrict__ imp,
                                                                 int64_t nhalves, int K,
                                                                 uint8_t *__restrict__ out) {
    const int64_t h = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= nhalves) return;
    const int64_t blk = h >> 1, half = h & 1;
    // sigma^2 over the whole block, summed in index order
    const float4 *b4 = reinterpret_cast<const float4 *>(W + blk * 32);
    float xb[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 t = b4[i];
        xb[4 * i] = t.x;
        xb[4 * i + 1] = t.y;
        xb[4 * i + 2] = t.z;
        xb[4 * i + 3] = t.w;
    }
    double s2 = 0.0;
#pragma unroll
    for (int i = 0; i < 32; ++i) s2 = __dadd_rn(s2, __dmul_rn((double)xb[i], (double)xb[i]));
    const double sigma2 = __ddiv_rn(__dmul_rn(2.0, s2), 32.0);
    float x[16];
    double w[16];
    const int k0 = (int)((blk * 32) % K) + 16 * (int)half;  // column of element 0 of the half
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        x[i] = xb[16 * half + i];
        const double xx = __dmul_rn((double)x[i], (double)x[i]);
        w[i] = __dmul_rn((double)imp[k0 + i], __dsqrt_rn(__dadd_rn(sigma2, xx)));
    }
    int best = 0;
    double best_sse = 0.0;
    for (int b = 0; b <= 0x7E; ++b) {
        const float s = ue4m3_scale(b);
        double sse = 0.0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float r = __fmul_rn(level_of(code_of(x[i], s)), s);
            const double e = __dsub_rn((double)x[i], (double)r);
            sse = __dadd_rn(sse, __dmul_rn(w[i], __dmul_rn(e, e)));
        }
        if (b == 0 || sse < best_sse) {
            best_sse = sse;
            best = b;
        }
    }
    const float s = ue4m3_scale(best);
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) word |= (uint32_t)code_of(x[i], s) << (2 * i);
    uint8_t *o = out + blk * 10;
#pragma unroll
    for (int i = 0; i < 4; ++i) o[4 * half + i] = (uint8_t)(word >> (8 * i));
    o[8 + half] = (uint8_t)best;
}

// Scale bytes >= 0x7F.
__global__ void rfp2_validate_kernel(const uint8_t *__restrict__ W, int64_t nblocks,
                                     unsigned long long *bad, int32_t *status) {
    unsigned long long local = 0;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < nblocks;
         j += (int64_t)gridDim.x * blockDim.x) {
        local += (W[j * 10 + 8] > 0x7E) + (W[j * 10 + 9] > 0x7E);
    }
    if (local) {
        atomicAdd(bad, local);
        record_status(status, RFP2_EBADSCALE);
    }
}

// Every int32 half sum with the GEMV's own expansion code.
__global__ void half_partials_kernel(const uint8_t *__restrict__ W, int M, int K,
                                     const int8_t *__restrict__ q, int N,
                                     int32_t *__restrict__ partials) {
    const int KB = K >> 5;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (int64_t)N * M * KB) return;
    const int j = (int)(t % KB);
    const int64_t nm = t / KB;
    const int m = (int)(nm % M), n = (int)(nm / M);
    const uint8_t *blk = W + ((int64_t)m * KB + j) * 10;
    const uint32_t lo = blk[0] | (blk[1] << 8) | (blk[2] << 16) | ((uint32_t)blk[3] << 24);
    const uint32_t hi = blk[4] | (blk[5] << 8) | (blk[6] << 16) | ((uint32_t)blk[7] << 24);
    const uint4 *qa = reinterpret_cast<const uint4 *>(q + (int64_t)n * K + (int64_t)j * 32);
    const uint4 x0 = qa[0], x1 = qa[1];
    uint32_t a0[4], a1[4], w0[4], w1[4];
    permute_act_half(x0.x, x0.y, x0.z, x0.w, a0);
    permute_act_half(x1.x, x1.y, x1.z, x1.w, a1);
    expand_half(lo, w0);
    expand_half(hi, w1);
    int32_t *o = partials + nm * (K / 16) + 2 * j;
    o[0] = half_dot_biased(w0, a0) - kDotBias;
    o[1] = half_dot_biased(w1, a1) - kDotBias;
}

// Nearest E2M1 magnitude index of a >= 0 (a <= 6 by construction), ties to
// the even index: thresholds are the midpoints of adjacent magnitudes; the
// comparison is >= where the upper neighbour has the even index.
__device__ __forceinline__ int e2m1_index(double a) {
    return (a > 0.25) + (a >= 0.75) + (a > 1.25) + (a >= 1.75) + (a > 2.5) + (a >= 3.5) +
           (a > 5.0);
}

// One CTA (256 threads) per HFP4 row.
__global__ void __launch_bounds__(256) hfp4_pack_kernel(const float *__restrict__ W, int K,
                                                        uint8_t *__restrict__ out,
                                                        int32_t *status) {
    __shared__ float wmax[8];
    const int64_t m = blockIdx.x;
    const float *w = W + m * (int64_t)K;
    const int64_t rb = 16 + 17 * (int64_t)(K / 32);
    uint8_t *row = out + m * rb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float amax = 0.0f;
    for (int k = threadIdx.x; k < K; k += blockDim.x) amax = fmaxf(amax, fabsf(w[k]));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) wmax[warp] = amax;
    __syncthreads();
    amax = 0.0f;
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, wmax[i]);
    const __half rs16 = __float2half_rn(__fdiv_rn(amax, 6.0f));
    const float rs = __half2float(rs16);
    if (!isfinite(rs)) {
        if (threadIdx.x == 0) record_status(status, RFP2_EINVAL);
    }
    if (threadIdx.x < 16) {
        const uint16_t bits = __half_as_ushort(rs16);
        const int nb = K / 32;
        uint8_t v = 0;
        if (threadIdx.x == 0) v = bits & 0xFF;
        if (threadIdx.x == 1) v = bits >> 8;
        if (threadIdx.x == 4) v = nb & 0xFF;
        if (threadIdx.x == 5) v = (nb >> 8) & 0xFF;
        row[threadIdx.x] = v;
    }
    for (int j = warp; j < K / 32; j += 8) {
        const float x = w[j * 32 + lane];
        const float wn = (rs == 0.0f) ? 0.0f : __fdiv_rn(x, rs);
        float bmax = fabsf(wn);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
            bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, off));
        // smallest e in [0, 254] with bmax <= 6 * 2^(e - 127)
        const double bm = (double)bmax;
        int e = 0;
        if (bm > 0.0) {
            e = ilogb(bm) - 2 + 127;
            if (e < 0) e = 0;
            if (e > 254) e = 254;
            while (e > 0 && bm <= 6.0 * ldexp(1.0, e - 1 - 127)) --e;
            while (e < 254 && !(bm <= 6.0 * ldexp(1.0, e - 127))) ++e;
        }
        const double v = ldexp((double)wn, 127 - e);
        const int code = e2m1_index(fabs(v)) | (signbit(wn) ? 8 : 0);
        // pair up even/odd lanes into one byte (low nibble = even index)
        const int other = __shfl_xor_sync(0xffffffffu, code, 1);
        uint8_t *blk = row + 16 + 17 * (int64_t)j;
        if ((lane & 1) == 0) blk[1 + lane / 2] = (uint8_t)(code | (other << 4));
        if (lane == 0) blk[0] = (uint8_t)e;
    }
}

}  // namespace
}  // namespace rfp2

using namespace rfp2;

extern "C" rfp2_status rfp2_pack_weights(const float *W, int64_t M, int64_t K, uint8_t *out,
                                         rfp2_stream_t stream) {
    if (M < 0 || K < 0) return RFP2_EINVAL;
    if (K % 32 != 0) return RFP2_ESHAPE;
    if (M == 0 || K == 0) return RFP2_OK;
    if (!W || !out) return RFP2_EINVAL;
    if (!aligned(W, 16)) return RFP2_EALIGN;
    const int64_t nh = M * K / 16;
    const int64_t ctas = (nh + 255) / 256;
    if (ctas > 0x7FFFFFFF) return RFP2_ESHAPE;
    return from_cuda(launch(rfp2_pack_kernel, dim3((unsigned)ctas), dim3(256), 0,
                            reinterpret_cast<cudaStream_t>(stream), false, W, nh, out));
}

extern "C" rfp2_status rfp2_pack_weights_weighted(const float *W, int64_t M, int64_t K,
                                                  const float *importance, uint8_t *out,
                                                  rfp2_stream_t stream) {
    if (M < 0 || K < 0) return RFP2_EINVAL;
    if (K % 32 != 0 || K > 0x7FFFFFFF) return RFP2_ESHAPE;
    if (M == 0 || K == 0) return RFP2_OK;
    if (!W || !importance || !out) return RFP2_EINVAL;
    if (!aligned(W, 16) || !aligned(importance, 4)) return RFP2_EALIGN;
    const int64_t nh = M * K / 16;
    const int64_t ctas = (nh + 255) / 256;
    if (ctas > 0x7FFFFFFF) return RFP2_ESHAPE;
    return from_cuda(launch(rfp2_pack_weighted_kernel, dim3((unsigned)ctas), dim3(256), 0,
                            reinterpret_cast<cudaStream_t>(stream), false, W, importance, nh,
                            (int)K, out));
}

extern "C" rfp2_status hfp4_pack_weights(const float *W, int64_t M, int64_t K, uint8_t *out,
                                         int32_t *dev_status, rfp2_stream_t stream) {
    if (M < 0 || K < 0) return RFP2_EINVAL;
    if (K % 32 != 0 || K / 32 > 0xFFFF || M > 0x7FFFFFFF) return RFP2_ESHAPE;
    if (M == 0 || K == 0) return RFP2_OK;
    if (!W || !out) return RFP2_EINVAL;
    if (!aligned(W, 4)) return RFP2_EALIGN;
    return from_cuda(launch(hfp4_pack_kernel, dim3((unsigned)M), dim3(256), 0,
                            reinterpret_cast<cudaStream_t>(stream), false, W, (int)K, out,
                            dev_status));
}

extern "C" rfp2_status rfp2_validate_weights(const uint8_t *W, int64_t nblocks,
                                             int64_t *bad_count, int32_t *dev_status,
                                             rfp2_stream_t stream) {
    if (nblocks < 0 || !bad_count) return RFP2_EINVAL;
    if (nblocks == 0) return RFP2_OK;
    if (!W) return RFP2_EINVAL;
    if (!aligned(bad_count, 8)) return RFP2_EALIGN;
    int64_t ctas = (nblocks + 255) / 256;
    const int64_t cap = 4LL * sm_count(current_device());
    if (ctas > cap) ctas = cap;
    return from_cuda(launch(rfp2_validate_kernel, dim3((unsigned)ctas), dim3(256), 0,
                            reinterpret_cast<cudaStream_t>(stream), false, W, nblocks,
                            reinterpret_cast<unsigned long long *>(bad_count), dev_status));
}

extern "C" rfp2_status rfp2_debug_half_partials(const uint8_t *W, int64_t M, int64_t K,
                                                const int8_t *q, int64_t N, int32_t *partials,
                                                rfp2_stream_t stream) {
    if (M <= 0 || K <= 0 || N <= 0) return RFP2_ESHAPE;
    if (K % 32 != 0 || M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF) return RFP2_ESHAPE;
    if (!W || !q || !partials) return RFP2_EINVAL;
    if (!aligned(q, 16)) return RFP2_EALIGN;
    const int64_t total = N * M * (K / 32);
    const int64_t ctas = (total + 255) / 256;
    if (ctas > 0x7FFFFFFF) return RFP2_ESHAPE;
    return from_cuda(launch(half_partials_kernel, dim3((unsigned)ctas), dim3(256), 0,
                            reinterpret_cast<cudaStream_t>(stream), false, W, (int)M, (int)K, q,
                            (int)N, partials));
}

namespace rfp2 {
namespace {

// One thread waits, with the library's bounded mbarrier wait, on a barrier
// that nothing ever arrives on: the wait gives up after the time limit and
// the kernel reports RFP2_ETIMEOUT, as every pipeline kernel does when a
// partner stops.
__global__ void debug_wait_kernel(int32_t *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        if (!mbar_wait(&bar, 0)) record_status(status, RFP2_ETIMEOUT);
    }
}

}  // namespace
}  // namespace rfp2

extern "C" rfp2_status rfp2_debug_wait_timeout(int32_t *dev_status, rfp2_stream_t stream) {
    if (!dev_status) return RFP2_EINVAL;
    if (!rfp2::aligned(dev_status, 4)) return RFP2_EALIGN;
    return rfp2::from_cuda(rfp2::launch(rfp2::debug_wait_kernel, dim3(1), dim3(32), 0,
                                        reinterpret_cast<cudaStream_t>(stream), false, dev_status));
}
