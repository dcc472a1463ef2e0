// ROCmFP2 weights decoded exactly to a 16-bit float type ("ROCmFP2 codebook
// research report", section "02 Quantization": a codebook level times a UE4M3
// scale has at most 4 significant bits and lies in [2^-10, 960] or is 0, so
// bf16 and f16 both hold it exactly).  Used by the prefill GEMM's decode
// warps, which write the values straight into the tensor cores' B stages.
#pragma once

#include <stdint.h>

#include "common.cuh"
#include "rfp2_decode.cuh"

namespace rfp2 {
namespace {

// The 16 weights of one half (code word c, weight i in bits 2i..2i+1; scale s,
// exact in bf16) -> eight words of two bf16 values, weights 2p and 2p+1 in
// word p (low, high).  All four levels {-4s, -s, s, 4s} share the low byte
// of bf16(s) (times 4 adds 2 to the exponent, leaving its lowest bit), so a
// PRMT over a table of their four high bytes gives every high byte, and one
// more PRMT plus an AND-OR puts each pair of weights together.  s = 0 gives
// -0 / +0 like level * s does.
RFP2_DEV void decode_half_bf16(uint32_t c, float s, uint32_t (&v)[8]) {
    const uint32_t sb = __float_as_uint(s) >> 16;      // bf16(s)
    const uint32_t hs = sb >> 8, h4 = hs + (sb != 0);  // high bytes of s and 4s
    // table bytes for codes 0..3: -4s, -s, s, 4s
    const uint32_t T = h4 * 0x01000001u + hs * 0x00010100u + 0x00008080u;
    const uint32_t lo = (sb & 0xFFu) * 0x00010001u;  // the shared low byte, both lanes
    const uint32_t m = c & 0x33333333u, n = (c >> 2) & 0x33333333u;
    // high bytes of the even weights [0 2 4 6], [8 10 12 14] and odd ones
    const uint32_t e0 = __byte_perm(T, 0u, m), e1 = __byte_perm(T, 0u, m >> 16);
    const uint32_t o0 = __byte_perm(T, 0u, n), o1 = __byte_perm(T, 0u, n >> 16);
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const uint32_t q = (uint32_t)(p & 3);
        const uint32_t x = __byte_perm(p < 4 ? e0 : e1, p < 4 ? o0 : o1,
                                       q | (q << 4) | ((4 + q) << 8) | ((4 + q) << 12));
        v[p] = (x & 0xFF00FF00u) | lo;
    }
}

}  // namespace
}  // namespace rfp2
