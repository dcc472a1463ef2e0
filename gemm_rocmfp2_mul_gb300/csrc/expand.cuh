// ROCmFP2 weights expanded to a 16-bit float type, one thread per 32-weight
// block ("ROCmFP2 codebook research report", section "02 Quantization": a
// codebook level times a UE4M3 scale has at most 4 significant bits and lies
// in [2^-10, 960] or is 0, so bf16 and f16 both hold it exactly).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"
#include "rfp2_decode.cuh"

namespace rfp2 {
namespace {

// Per output type: the 16-bit float whose low byte is an integer 0..255
// added to a power of two with unit spacing (f16 1024 = 0x6400, bf16 128 =
// 0x4300), and the bias that, subtracted, leaves the codebook level.
template <typename T>
struct Lanes;
template <>
struct Lanes<__half> {
    using T2 = __half2;
    static constexpr uint32_t kMagic = 0x64006400u;  // 1024 in both halves
    static __device__ __forceinline__ T2 bias() { return __float2half2_rn(1028.0f); }
    static __device__ __forceinline__ T2 splat(float v) { return __float2half2_rn(v); }
    static __device__ __forceinline__ uint32_t bits(T2 v) { return *reinterpret_cast<uint32_t *>(&v); }
    static __device__ __forceinline__ T2 from_bits(uint32_t b) { return *reinterpret_cast<T2 *>(&b); }
};
template <>
struct Lanes<__nv_bfloat16> {
    using T2 = __nv_bfloat162;
    static constexpr uint32_t kMagic = 0x43004300u;  // 128 in both halves
    static __device__ __forceinline__ T2 bias() { return __float2bfloat162_rn(132.0f); }
    static __device__ __forceinline__ T2 splat(float v) { return __float2bfloat162_rn(v); }
    static __device__ __forceinline__ uint32_t bits(T2 v) { return *reinterpret_cast<uint32_t *>(&v); }
    static __device__ __forceinline__ T2 from_bits(uint32_t b) { return *reinterpret_cast<T2 *>(&b); }
};

// Codebook levels plus 4 (-4, -1, +1, +4 -> 0, 3, 5, 8) as PRMT table bytes.
constexpr uint32_t kBiasedCodebookWord = 0x08050300u;

// One thread per 32-weight block.  The 16 selectors of a half become four
// words of biased levels with the same mask/shift/PRMT steps as the GEMV
// decode; a PRMT then pairs two neighbouring weights into the low bytes of
// a 2 x 16-bit word, the magic high byte turns each into (2^p + level + 4),
// one packed subtract leaves the level and one packed multiply by the scale
// gives level * scale: exact in both types, the rounding never acts.
template <typename T>
__global__ void __launch_bounds__(256) expand_kernel(const uint8_t *__restrict__ W,
                                                     int64_t nblocks, T *__restrict__ out) {
    using L = Lanes<T>;
    pdl_wait();
    pdl_launch_dependents();
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= nblocks) return;
    // the 10-byte block at byte 10j: one 16-bit and two aligned 32-bit loads,
    // all inside the block (10j is even; either 10j or 10j + 2 is 4-aligned)
    const uint8_t *b = W + j * 10;
    uint32_t lo, hi, pair;
    if ((j & 1) == 0) {  // 10j % 4 == 0
        const uint32_t *w = reinterpret_cast<const uint32_t *>(b);
        lo = __ldg(w);
        hi = __ldg(w + 1);
        pair = __ldg(reinterpret_cast<const unsigned short *>(b + 8));
    } else {  // 10j % 4 == 2
        const uint32_t h0 = __ldg(reinterpret_cast<const unsigned short *>(b));
        const uint32_t *w = reinterpret_cast<const uint32_t *>(b + 2);
        const uint32_t w1 = __ldg(w), w2 = __ldg(w + 1);
        lo = h0 | (w1 << 16);
        hi = __funnelshift_r(w1, w2, 16);
        pair = w2 >> 16;
    }
    float s0, s1;
    decode_scale_pair(pair, s0, s1);
    const typename L::T2 bias = L::bias();
    uint4 *o = reinterpret_cast<uint4 *>(out + j * 32);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t c = h ? hi : lo;
        const typename L::T2 sc = L::splat(h ? s1 : s0);
        // lanes [0 2 4 6] [8 10 12 14] [1 3 5 7] [9 11 13 15] of the half
        const uint32_t m = c & 0x33333333u, n = (c >> 2) & 0x33333333u;
        uint32_t w[4];
        w[0] = __byte_perm(kBiasedCodebookWord, 0u, m);
        w[1] = __byte_perm(kBiasedCodebookWord, 0u, m >> 16);
        w[2] = __byte_perm(kBiasedCodebookWord, 0u, n);
        w[3] = __byte_perm(kBiasedCodebookWord, 0u, n >> 16);
        uint32_t v[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) {  // weights 2p, 2p+1 of the half
            const uint32_t x = __byte_perm(p < 4 ? w[0] : w[1], p < 4 ? w[2] : w[3],
                                           (uint32_t)((p & 3) | ((4 + (p & 3)) << 8)));
            const typename L::T2 t = L::from_bits((x & 0x00FF00FFu) | L::kMagic);
            v[p] = L::bits(__hmul2(__hsub2(t, bias), sc));
        }
        o[2 * h] = make_uint4(v[0], v[1], v[2], v[3]);
        o[2 * h + 1] = make_uint4(v[4], v[5], v[6], v[7]);
    }
}

}  // namespace
}  // namespace rfp2
