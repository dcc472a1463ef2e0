// Dense ROCmFP2 GEMV: y[n, m] = sum_k w[m, k] * q[n, k] * dA (int8 path).
//
// Source: "ROCmFP2 codebook research report", sections "01 Storage",
// "02 Quantization" and "03 Runtime" (LOAD -> SPREAD -> PERMUTE -> DOT4 ->
// RESCALE, with each block expanded once for every activation column).
//
// GB300 design.  The packed weights (2.5 bits per weight) are the only large
// stream.  The block decode is bound by the integer pipe (about 23 ALU
// instructions per block and lane: mask, shifts, PRMTs, scale placement).
// A call's activations may only be read once the kernel before it has
// completed, so everything between that release and the first dot product
// (reading x, quantizing it, publishing it to every warp) lies on the
// critical path of every call and is kept short.
//  * Persistent grid, one CTA per SM, two CTAs resident per SM: the next
//    call's CTA becomes resident as soon as this one starts
//    (griddepcontrol.launch_dependents at entry), so its weight stream can
//    overlap this call (when weight prefetch is enabled; see
//    rfp2_set_weight_prefetch) and its barriers are ready when this call ends.
//  * CTA i owns the contiguous rows [i*M/G, (i+1)*M/G).  A producer warp
//    streams them in stages of R*RGS rows with 1-D bulk async copies (L2
//    evict-first) into a ring of as many stages as fit beside the quantized
//    activations; the rows beyond the ring are prefetched into L2 at entry.
//    The consumer warps form H sets that take alternate stages (set h takes
//    stages h, h + H, ...), so a stage is a small unit of the ring (about
//    20 KB) while every warp still decodes two rows per stage.
//  * Each CTA reads x straight from global memory after the release (no
//    staging copy) and quantizes it (Q8_1-style, bit-exact): four lanes per
//    32-value block, eight values per lane.  The int8 values go to shared
//    memory already permuted into the lane order of expand_half, one 16-byte
//    word per lane and half-block at an offset that is a compile-time
//    constant from a per-lane base, so the decode loop reads them with
//    conflict-free 16-byte loads and no address arithmetic.
//  * A warp reduces its rows' lane partials across the warp with a
//    transposing butterfly and stores them: after every three stages at one
//    column and every two at two columns (the partials wait in registers, so
//    the warp does not stall on the shuffle latency after each stage), else
//    after every stage.  Rows
//    split over several warps along K (very long rows) are combined through
//    a double-buffered shared-memory slot guarded by mbarriers.
//  * Every wait is an mbarrier wait with a time limit; a timeout stores
//    RFP2_ETIMEOUT and the CTA winds down after its copies have landed.
#include <mutex>

#include <algorithm>

#include "common.cuh"
#include "gemv_core.cuh"
#include "quantize.cuh"

namespace rfp2 {
namespace {

// Launch shapes: two CTAs per SM; CW consumer warps + 1 producer warp, each
// consumer decoding kRows rows of a stage at once.  Up to three columns: 16
// warps of at most 56 registers, four per SM sub-partition to hide each
// other's latencies (three columns spill a few registers and still gain,
// measured).  From four columns the extra activation and accumulator
// registers would spill heavily at 56, so 8 warps of up to 112 registers.
#ifndef RFP2_GEMV_WIDE_CW
#define RFP2_GEMV_WIDE_CW 8
#endif
#ifndef RFP2_GEMV_DEFER
#define RFP2_GEMV_DEFER 3
#endif
template <int NC>
constexpr int cw_of() {
    return NC <= 3 ? 16 : RFP2_GEMV_WIDE_CW;
}
constexpr int kRows = 2;
// Values (rows x columns) a warp reduces per stage, padded to a power of two.
constexpr int kVMax = 16;
// Stages whose partials a warp keeps in registers before one reduction
// covers them all (a warp owning whole rows; 1: reduce after every stage).
// At one column the three stages a set decodes at the 14336 x 4096 decode
// shape are reduced together, at two columns pairs of stages; from three
// columns the partials would spill.
template <int NC>
constexpr int defer_of() {
    return NC == 1 ? RFP2_GEMV_DEFER : NC == 2 ? 2 : 1;
}
// Shared memory per CTA: two CTAs per SM, or one when a shape needs more.
constexpr size_t kSmemPair = 113 * 1024;
constexpr size_t kSmemOne = 227 * 1024;
constexpr int kMaxStages = 32;
// Largest batch quantized inside the GEMV kernel by every CTA.
constexpr int64_t kFusedMaxN = 8;

// Activation groups (eight blocks of one column) a warp quantizes per pass:
// the K = 4096 case spread over the consumer warps, at most four in flight.
template <int NC, int CW>
constexpr int act_groups_per_pass() {
    return 16 * NC / CW < 1 ? 1 : 16 * NC / CW > 4 ? 4 : 16 * NC / CW;
}

struct GsArgs {
    const uint8_t *W;
    const int8_t *q;  // pre-quantized activations (FQ = false)
    const float *d;
    const float *x;   // fp32 activations (FQ = true)
    int8_t *qout;     // optional copies of q/d in natural layout (FQ, CTA 0)
    float *dout;
    float *y;
    int32_t *status;
    int M, K, WK, H, stages, rows_per_cta, rows_extra, x_vec, w_early;
    uint32_t off_bars, off_red, off_actq, off_actd;
};

// ---------------------------------------------------------------------------
// Activations in shared memory.  Block kb of column n sits with the lane
// that decodes it: K-slice wk = kb / (32*BPT), lane l = (kb / BPT) % 32,
// b = kb % BPT.  Its 32 int8 values are two 16-byte words (h = 0, 1: the
// halves) at word index (((wk*BPT + b)*2 + h)*NC + n)*32 + l, and its scale
// dA (times 2^19, see block_sum_2m19) is float ((wk*BPT + b)*NC + n)*32 + l.
// The 16 values of a half are stored as [a0 a2 a4 a6 | a1 a3 a5 a7 | a8 a10
// a12 a14 | a9 a11 a13 a15] (even and odd positions of each group of eight);
// the decode reorders the four words into the lane order of expand_half.
// For fixed (b, h, n) the 32 lanes read 512 consecutive bytes: no bank
// conflicts, and a lane's offsets from its base are compile-time constants.

RFP2_DEV uint32_t act_word_index(int wk, int b, int h, int n, int l, int BPT, int NC) {
    return ((((uint32_t)wk * BPT + b) * 2 + h) * NC + n) * 32 + l;
}

// Bytes 0 of a, b -> bytes 0, 1 of the result.
RFP2_DEV uint32_t lo_bytes(uint32_t a, uint32_t b) { return prmt(a, b, 0x0040u); }
// Four values (low byte of each word) -> one word, first value in byte 0.
RFP2_DEV uint32_t pack4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    return prmt(lo_bytes(a, b), lo_bytes(c, d), 0x5410u);
}

RFP2_DEV float rcp_approx_f(float v) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// Scales from which the near-half rounding below is exact (every product and
// residual in it stays a normal float).
constexpr float kExactHalfMinD = 0x1p-100f;

// roundf(fl(a / d)) for a value whose quotient estimate z (|z - a/d| <
// 2^-14) lies within 2^-12 of a half-integer, for d >= kExactHalfMinD,
// decided without a division.  With A = |a| and H = floor(|z|) + 1/2 that
// half-integer, fl(A/d) >= H (roundf then goes away from zero) exactly when
// A/d >= H - u/2, u being the float spacing just below H; at equality the
// even significand would win (a tie there needs A to carry 25 significant
// bits, so it never happens for float inputs; the test is kept all the same).
// R = A - H*d is a small multiple of d's quantum (|R| < 2^-11 d, and H has
// at most eight significant bits), so the FMA computes it exactly, and
// (u/2)*d is exact too (u/2 is a power of two): one comparison decides.
RFP2_DEV float round_quotient_near_half(float a, float d, float z) {
    const float A = fabsf(a);
    const float H = floorf(fabsf(z)) + 0.5f;
    const float R = fmaf(-H, d, A);
    const uint32_t hb = __float_as_uint(H);
    // u/2: 2^(e-24) for H in (2^e, 2^(e+1)); 2^(e-25) when H = 2^e (H = 0.5)
    const uint32_t drop = (hb & 0x7FFFFFu) == 0u ? 25u : 24u;
    const float half_u = __uint_as_float(((hb >> 23) - drop) << 23);
    const float t = half_u * d;
    const bool up = R > -t || (R == -t && (hb & 1u) == 0u);
    return copysignf((H - 0.5f) + (up ? 1.0f : 0.0f), a);
}

// Work split of the activation pass: a group is eight blocks of one column
// that eight consecutive lanes l of one K-slice decode (same b), four
// quantizing lanes per block and eight values per lane.  Group gi of a
// column-major enumeration: o = gi % 4 (lanes 8o .. 8o+7), then b, then wk,
// then n.  WK and BPT are powers of two.
struct ActSlot {
    int n, wk, b, l, kb;
};
template <int BPT>
RFP2_DEV ActSlot act_slot(int gi, int lane, int log_wk, int WK) {
    constexpr int LB = Log2<BPT>::v;
    ActSlot s;
    const int t = gi >> 2;
    s.b = t & (BPT - 1);
    const int t2 = t >> LB;
    s.wk = t2 & (WK - 1);
    s.n = t2 >> log_wk;
    s.l = 8 * (gi & 3) + (lane >> 2);
    s.kb = (s.wk * 32 + s.l) * BPT + s.b;
    return s;
}

// Quantize the NC x K activations (global x) into the permuted shared layout;
// CTA 0 also writes q and d in natural layout to gq/gd.  Same results as the
// quantize kernel (d = amax / 127 and q = roundf(a / d), IEEE divisions): q
// comes from z = a * rcp.approx(d), whose relative error is below 2^-22, so
// |z - a/d| < 2^-14 (|a/d| <= 127) and the IEEE quotient fl(a/d) lies within
// 2^-17 of a/d.  Both therefore round to the same integer unless z is within
// 2^-12 of a half-integer; those values are rounded by an exact comparison
// (round_quotient_near_half), or, where d is tiny (and z may not even be
// finite: a subnormal d whose reciprocal overflows), by the IEEE division and
// roundf.
// Elsewhere z + 1.5*2^23 rounds z to that integer and holds it, in two's
// complement, in the low byte of its bits.
template <int NC, int BPT, int QP, int CW>
RFP2_DEV void quantize_to_smem(const float *__restrict__ x, bool vec, int K, int WK, int log_wk,
                               int warp, int lane, uint8_t *actq, float *actd, int8_t *gq,
                               float *gd) {
    const int KB = K >> 5;
    const int ngroups = NC * WK * BPT * 4;
    const int quarter = lane & 3, h = quarter >> 1, part = quarter & 1;
    for (int g0 = warp; g0 < ngroups; g0 += CW * QP) {
        float v[QP][8];
        ActSlot s[QP];
        bool in[QP], ok[QP];
#pragma unroll
        for (int i = 0; i < QP; ++i) {
            const int gi = g0 + i * CW;
            in[i] = gi < ngroups;  // the same for the whole warp
            s[i] = act_slot<BPT>(in[i] ? gi : 0, lane, log_wk, WK);
            ok[i] = in[i] && s[i].kb < KB;
            const float *src = x + (size_t)s[i].n * K + (size_t)s[i].kb * 32 + quarter * 8;
            if (!ok[i]) {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[i][e] = 0.0f;
            } else if (vec) {
                const float4 t0 = *reinterpret_cast<const float4 *>(src);
                const float4 t1 = *reinterpret_cast<const float4 *>(src + 4);
                v[i][0] = t0.x, v[i][1] = t0.y, v[i][2] = t0.z, v[i][3] = t0.w;
                v[i][4] = t1.x, v[i][5] = t1.y, v[i][6] = t1.z, v[i][7] = t1.w;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[i][e] = src[e];
            }
        }
#pragma unroll
        for (int i = 0; i < QP; ++i) {
            float m = fabsf(v[i][0]);
#pragma unroll
            for (int e = 1; e < 8; ++e) m = fmaxf(m, fabsf(v[i][e]));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            const float d = __fdiv_rn(m, 127.0f);
            const float rc = d != 0.0f ? rcp_approx_f(d) : 0.0f;
            uint32_t qb[8];
            if constexpr (NC == 1) {
                // Every value also takes the exact near-half decision and
                // keeps it where z is near a half-integer: no branch, so no
                // warp waits on a division (every CTA waits for its slowest
                // warp).  Only scales too small for that decision (never in
                // practice) take the IEEE division.
                const bool exact_half = d >= kExactHalfMinD;
                uint32_t need = 0;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float z = v[i][e] * rc;
                    const float zb = z + 12582912.0f;
                    const float t = z - (zb - 12582912.0f);
                    const bool near = !(fabsf(t) <= 0.5f - 0x1p-12f);
                    const float r = round_quotient_near_half(v[i][e], d, z);
                    qb[e] = near && exact_half ? __float_as_uint(r + 12582912.0f) : __float_as_uint(zb);
                    need |= (near && !exact_half ? 1u : 0u) << e;
                }
                if (__any_sync(0xffffffffu, need != 0u) && need != 0u && d != 0.0f) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float qf = fminf(fmaxf(roundf(__fdiv_rn(v[i][e], d)), -127.0f), 127.0f);
                        if ((need >> e) & 1u) qb[e] = (uint32_t) static_cast<int>(qf);
                    }
                }
            } else {
                // several columns: the branch-free decision would cost more
                // than it saves (measured), so the lanes with a value near a
                // boundary take the IEEE division for all their values
                bool need = false;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float z = v[i][e] * rc;
                    const float zb = z + 12582912.0f;
                    const float t = z - (zb - 12582912.0f);
                    need |= !(fabsf(t) <= 0.5f - 0x1p-12f);
                    qb[e] = __float_as_uint(zb);
                }
                if (__any_sync(0xffffffffu, need) && need && d != 0.0f) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float qf = fminf(fmaxf(roundf(__fdiv_rn(v[i][e], d)), -127.0f), 127.0f);
                        qb[e] = (uint32_t) static_cast<int>(qf);
                    }
                }
            }
            if (!in[i]) continue;
            const uint32_t ev = pack4(qb[0], qb[2], qb[4], qb[6]);
            const uint32_t od = pack4(qb[1], qb[3], qb[5], qb[7]);
            const uint32_t wi = act_word_index(s[i].wk, s[i].b, h, s[i].n, s[i].l, BPT, NC);
            *reinterpret_cast<uint2 *>(actq + wi * 16 + part * 8) =
                ok[i] ? make_uint2(ev, od) : make_uint2(0u, 0u);
            if (quarter == 0)
                actd[(((size_t)s[i].wk * BPT + s[i].b) * NC + s[i].n) * 32 + s[i].l] =
                    ok[i] ? d * 0x1p19f : 0.0f;
            if (gq && ok[i]) {
                const size_t e0 = (size_t)s[i].n * K + (size_t)s[i].kb * 32 + quarter * 8;
                *reinterpret_cast<uint2 *>(gq + e0) = make_uint2(
                    pack4(qb[0], qb[1], qb[2], qb[3]), pack4(qb[4], qb[5], qb[6], qb[7]));
                if (quarter == 0) gd[(size_t)s[i].n * KB + s[i].kb] = d;
            }
        }
    }
}

// Pre-quantized q/d (natural layout, global memory) into the permuted shared
// layout, with the same work split.
template <int NC, int BPT, int QP, int CW>
RFP2_DEV void permute_to_smem(const int8_t *__restrict__ q, const float *__restrict__ d, int K,
                              int WK, int log_wk, int warp, int lane, uint8_t *actq,
                              float *actd) {
    const int KB = K >> 5;
    const int ngroups = NC * WK * BPT * 4;
    const int quarter = lane & 3, h = quarter >> 1, part = quarter & 1;
    for (int g0 = warp; g0 < ngroups; g0 += CW * QP) {
        uint2 w[QP];
        float dv[QP];
        ActSlot s[QP];
        bool in[QP], ok[QP];
#pragma unroll
        for (int i = 0; i < QP; ++i) {
            const int gi = g0 + i * CW;
            in[i] = gi < ngroups;
            s[i] = act_slot<BPT>(in[i] ? gi : 0, lane, log_wk, WK);
            ok[i] = in[i] && s[i].kb < KB;
            w[i] = ok[i] ? __ldg(reinterpret_cast<const uint2 *>(
                               q + (size_t)s[i].n * K + (size_t)s[i].kb * 32 + quarter * 8))
                         : make_uint2(0u, 0u);
            dv[i] = ok[i] ? __ldg(d + (size_t)s[i].n * KB + s[i].kb) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < QP; ++i) {
            if (!in[i]) continue;
            const uint32_t wi = act_word_index(s[i].wk, s[i].b, h, s[i].n, s[i].l, BPT, NC);
            *reinterpret_cast<uint2 *>(actq + wi * 16 + part * 8) =
                make_uint2(prmt(w[i].x, w[i].y, 0x6420u), prmt(w[i].x, w[i].y, 0x7531u));
            if (quarter == 0)
                actd[(((size_t)s[i].wk * BPT + s[i].b) * NC + s[i].n) * 32 + s[i].l] =
                    dv[i] * 0x1p19f;
        }
    }
}

// ---------------------------------------------------------------------------
// Decode of R rows (row_stride apart) against the activations: acc[r][n] +=
// sum over the lane's BPT blocks of dA*(d0*S0 + d1*S1), each block's sum
// formed as (d0*S0 + d1*S1) * 2^-19 by block_sum_2m19 and multiplied by the
// stored dA * 2^19.  The R rows share every activation load; abase/dbase are
// the lane's activation bases (its K-slice included).

template <int BPT>
RFP2_DEV void load_row_words(const uint8_t *p, uint32_t (&v)[BPT >= 2 ? 5 * BPT / 2 : 3]) {
    if constexpr (BPT == 8) {
        const uint4 *s = reinterpret_cast<const uint4 *>(p);
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            const uint4 t = s[i];
            v[4 * i] = t.x;
            v[4 * i + 1] = t.y;
            v[4 * i + 2] = t.z;
            v[4 * i + 3] = t.w;
        }
    } else if constexpr (BPT == 4) {
        const uint2 *s = reinterpret_cast<const uint2 *>(p);
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            const uint2 t = s[i];
            v[2 * i] = t.x;
            v[2 * i + 1] = t.y;
        }
    } else if constexpr (BPT == 2) {
        const uint32_t *s = reinterpret_cast<const uint32_t *>(p);
#pragma unroll
        for (int i = 0; i < 5; ++i) v[i] = s[i];
    } else {
        // one 10-byte block at a 2-byte aligned address: five halfwords
        const uint16_t *s = reinterpret_cast<const uint16_t *>(p);
        v[0] = (uint32_t)s[0] | ((uint32_t)s[1] << 16);
        v[1] = (uint32_t)s[2] | ((uint32_t)s[3] << 16);
        v[2] = (uint32_t)s[4];
    }
}

template <int BPT>
RFP2_DEV Block block_of(const uint32_t (&v)[BPT >= 2 ? 5 * BPT / 2 : 3], int b) {
    if constexpr (BPT == 1) {
        Block k;
        k.lo = v[0];
        k.hi = v[1];
        k.scales = v[2];
        return k;
    } else {
        return block_from_words<BPT>(v, b);
    }
}

template <int NC, int BPT, int R>
RFP2_DEV void decode_rows(const uint8_t *p0, uint32_t row_stride, const uint8_t *abase,
                          const float *dbase, float (&acc)[R][NC]) {
    constexpr int NW = BPT >= 2 ? 5 * BPT / 2 : 3;
    uint32_t v[R][NW];
#pragma unroll
    for (int r = 0; r < R; ++r) load_row_words<BPT>(p0 + r * row_stride, v[r]);
#pragma unroll
    for (int b = 0; b < BPT; ++b) {
        uint32_t wlo[R][4], whi[R][4];
        float s0[R], s1[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const Block k = block_of<BPT>(v[r], b);
            expand_half(k.lo, wlo[r]);
            expand_half(k.hi, whi[r]);
            placed_scale_pair(k.scales, s0[r], s1[r]);
        }
#pragma unroll
        for (int n = 0; n < NC; ++n) {
            const uint4 q0 = *reinterpret_cast<const uint4 *>(abase + ((b * 2 + 0) * NC + n) * 512);
            const uint4 q1 = *reinterpret_cast<const uint4 *>(abase + ((b * 2 + 1) * NC + n) * 512);
            const float dA = dbase[(b * NC + n) * 32];
            // stored [even lo | odd lo | even hi | odd hi] -> expand_half's order
            const uint32_t lo[4] = {q0.x, q0.z, q0.y, q0.w};
            const uint32_t hi[4] = {q1.x, q1.z, q1.y, q1.w};
#pragma unroll
            for (int r = 0; r < R; ++r)
                acc[r][n] = fmaf(block_sum_2m19(wlo[r], whi[r], s0[r], s1[r], lo, hi), dA, acc[r][n]);
        }
    }
}

// ---------------------------------------------------------------------------
// The kernel.  FQ: quantize x inside the kernel; otherwise q/d come
// pre-quantized from global memory.
template <int NC, int BPT, bool FQ>
__global__ void __launch_bounds__((cw_of<NC>() + 1) * 32, 2) gemv_stream_kernel(const GsArgs a) {
    constexpr int kCW = cw_of<NC>();
    constexpr int V = NextPow2<kRows * NC>::v;
    constexpr int L = Log2<V>::v;
    extern __shared__ __align__(128) uint8_t smem[];
    // let the next call's grid become resident at once (beside this CTA); it
    // touches x, y and the workspace only after this grid has completed
    pdl_launch_dependents();
    const int KB = a.K >> 5;
    const uint32_t rowbytes = (uint32_t)KB * 10;
    const int S = a.stages, H = a.H, WK = a.WK;
    const int G = kCW / H;       // warps per set
    const int RGS = G / WK;      // row groups per set
    const int SR = kRows * RGS;  // rows per stage
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.off_bars);
    uint64_t *empty = full + S;
    uint64_t *act_bar = empty + S;
    uint64_t *redfull = act_bar + 1;        // [kCW][2] (row-group id, parity)
    uint64_t *redfree = redfull + 2 * kCW;  // [kCW][2]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(redfree + 2 * kCW);
    float *red = reinterpret_cast<float *>(smem + a.off_red);  // [row group][2][WK][kVMax]
    uint8_t *actq = smem + a.off_actq;
    float *actd = reinterpret_cast<float *>(smem + a.off_actd);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bx = blockIdx.x;
    const int64_t r_begin = (int64_t)bx * a.rows_per_cta + min(bx, a.rows_extra);
    const int nrows = a.rows_per_cta + (bx < a.rows_extra ? 1 : 0);
    const int nstages = (nrows + SR - 1) / SR;
    const uint32_t stage_bytes = (uint32_t)SR * rowbytes;
    const uint8_t *src = a.W + r_begin * rowbytes;

    // Ring slots belong to the sets: set h owns slots h, h + H, ... < S, so
    // every use of a slot is consumed by the same set, in order (a parity
    // wait then always refers to the right round).  Stage c = h + H*j goes
    // to slot h + H*(j % S_h), round j / S_h.
    auto slot_of = [&](int c, int &round) {
        const int h = c % H, j = c / H;
        const int sh = (S - h + H - 1) / H;
        round = j / sh;
        return h + H * (j % sh);
    };
    auto stage_len = [&](int c) { return (uint32_t)min(SR, nrows - c * SR) * rowbytes; };
    auto issue = [&](int c, uint64_t pol) {
        int round;
        const int s = slot_of(c, round);
        mbar_arrive_expect_tx(&full[s], stage_len(c));
        bulk_g2s_stream(smem + (size_t)s * stage_bytes, src + (size_t)c * stage_bytes, stage_len(c),
                        &full[s], pol);
    };

    if (threadIdx.x == kCW * 32) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], G);
        }
        mbar_init(act_bar, kCW);
        for (int i = 0; i < 2 * kCW; ++i) {
            mbar_init(&redfull[i], WK > 1 ? WK - 1 : 1);
            mbar_init(&redfree[i], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
        // rows beyond the ring: into L2 now (always safe, L2 is coherent), so
        // their copies into the ring later are short
        for (int c = S; c < nstages; ++c) bulk_prefetch_l2(src + (size_t)c * stage_bytes, stage_len(c));
        if (a.w_early) {
            const uint64_t pol = policy_evict_first();
            for (int c = 0; c < nstages && c < S; ++c) issue(c, pol);
        }
    }
    __syncthreads();

    if (warp == kCW) {
        // ---- producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            pdl_wait();  // the earlier work (W unless prefetching) is complete
            int c = 0;
            if (a.w_early) {
                c = min(nstages, S);
            } else {
                for (; c < nstages && c < S; ++c) issue(c, pol);
            }
            for (; c < nstages; ++c) {
                int round;
                const int s = slot_of(c, round);
                if (!mbar_wait_sleepy(&empty[s], (round - 1) & 1)) {
                    record_status(a.status, RFP2_ETIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                issue(c, pol);
            }
            // No copy may still be in flight when the CTA exits.  Without an
            // abort every issued stage is waited for by its consumer set
            // before the CTA can exit, so the producer leaves at once (a
            // drain here was measured to hold the CTA up to ~0.8 us after
            // its last consumer).  After an abort (a wait ran out; consumers
            // may have left early) it waits for the latest round issued into
            // each slot of the first c stages.
            if (*abort_flag == 0) return;
            for (int s = 0; s < S; ++s) {
                const int h = s % H, jj = s / H, sh = (S - h + H - 1) / H;
                if (c <= h) continue;
                const int jmax = (c - 1 - h) / H;  // last issued stage index of set h
                if (jmax < jj) continue;           // slot never used
                const int j = jmax - (jmax - jj) % sh;
                if (!mbar_wait(&full[s], (j / sh) & 1)) record_status(a.status, RFP2_ETIMEOUT);
            }
        }
        return;
    }

    // ---- consumers: the activations into shared memory, then the stages
    const int log_wk = __ffs(WK) - 1;
    constexpr int QP = act_groups_per_pass<NC, kCW>();
    // The warp's place in the CTA.  At one column it is worked out before the
    // dependency wait (it does not depend on the earlier work); with more
    // columns the quantize needs those registers, so it comes after.
    struct WarpPlace {
        int set, rg, wk;
        uint32_t row_off;
    };
    auto place_warp = [&]() {
        WarpPlace w;
        w.set = warp / G;
        const int g = warp - w.set * G;
        w.rg = g >> log_wk;
        w.wk = g & (WK - 1);
        const int kb = (w.wk * 32 + lane) * BPT;
        // a row past the CTA's last one still lies inside the stage: it is
        // computed from stale bytes and never stored
        w.row_off = (uint32_t)(w.rg * kRows) * rowbytes + (kb < KB ? (uint32_t)kb * 10 : 0u);
        return w;
    };
    WarpPlace wp;
    if constexpr (NC == 1) wp = place_warp();
    pdl_wait();
    if constexpr (FQ) {
        quantize_to_smem<NC, BPT, QP, kCW>(a.x, a.x_vec != 0, a.K, WK, log_wk, warp, lane, actq,
                                           actd, bx == 0 ? a.qout : nullptr, a.dout);
    } else {
        permute_to_smem<NC, BPT, QP, kCW>(a.q, a.d, a.K, WK, log_wk, warp, lane, actq, actd);
    }
    // one arrival per warp: __syncwarp orders the warp's stores before lane
    // 0's release-arrive, which publishes them to the waiting warps
    __syncwarp();
    if (lane == 0) mbar_arrive(act_bar);
    if (!mbar_wait(act_bar, 0)) {
        record_status(a.status, RFP2_ETIMEOUT);
        *abort_flag = 1;
        return;
    }

    if constexpr (NC != 1) wp = place_warp();
    const int set = wp.set, rg = wp.rg, wk = wp.wk;
    const int wid = set * RGS + rg;  // row-group id, < kCW / WK
    const int kb0 = (wk * 32 + lane) * BPT;
    const bool active = kb0 < KB;
    const uint8_t *abase = actq + ((size_t)wk * BPT * 2 * NC * 32 + lane) * 16;
    const float *dbase = actd + (size_t)wk * BPT * NC * 32 + lane;
    const uint32_t row_off = wp.row_off;
    int slot = set, phase = 0;  // the set's own slots: set, set + H, ... < S

    // the stage in `slot` is in shared memory (false: time limit or abort);
    // the abort flag is read only when the stage has not landed yet
    auto stage_ready = [&]() {
        if (mbar_try_wait(&full[slot], phase)) return true;
        if (*abort_flag || !mbar_wait(&full[slot], phase)) {
            record_status(a.status, RFP2_ETIMEOUT);
            *abort_flag = 1;
            return false;
        }
        return true;
    };
    auto next_slot = [&]() {
        slot += H;
        if (slot >= S) {
            slot = set;
            phase ^= 1;
        }
    };

    constexpr int D = defer_of<NC>();
    if (D > 1 && WK == 1) {
        // A warp owns whole rows: the lane partials of D consecutive stages
        // stay in registers and one transposing reduction covers them all,
        // so the warp does not stall on the reduction's shuffle latency
        // after every stage.
        constexpr int VS = kRows * NC;
        constexpr int VD = NextPow2<D * VS>::v;
        constexpr int LD = Log2<VD>::v;
        const int idx = lane >> (5 - LD);
        const bool writer = (lane & ((32 >> LD) - 1)) == 0 && idx < D * VS;
        const int vj = idx / VS, vr = (idx / NC) % kRows, vn = idx % NC;
        for (int c0 = set; c0 < nstages; c0 += D * H) {
            float part[D][kRows][NC];
#pragma unroll
            for (int j = 0; j < D; ++j)
#pragma unroll
                for (int r = 0; r < kRows; ++r)
#pragma unroll
                    for (int n = 0; n < NC; ++n) part[j][r][n] = 0.0f;
#pragma unroll
            for (int j = 0; j < D; ++j) {
                if (c0 + j * H < nstages) {
                    if (!stage_ready()) return;
                    if (active)
                        decode_rows<NC, BPT, kRows>(smem + (size_t)slot * stage_bytes + row_off,
                                                    rowbytes, abase, dbase, part[j]);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[slot]);
                    next_slot();
                }
            }
            float vals[VD];
#pragma unroll
            for (int i = 0; i < VD; ++i)
                vals[i] = i < D * VS ? part[i / VS][(i / NC) % kRows][i % NC] : 0.0f;
            const float total = warp_transpose_reduce<VD>(vals, lane);
            const int c = c0 + vj * H;
            const int row = c * SR + rg * kRows + vr;
            if (writer && c < nstages && row < nrows) a.y[(int64_t)vn * a.M + r_begin + row] = total;
        }
        return;
    }

    // this lane's value after the warp reduction: row vr, column vn
    const int idx = lane >> (5 - L);
    const bool writer = (lane & ((32 >> L) - 1)) == 0 && idx < kRows * NC;
    const int vr = idx / NC, vn = idx - vr * NC;
    int it = 0;  // stages this warp has done
    for (int c = set; c < nstages; c += H, ++it) {
        if (!stage_ready()) return;
        float acc[kRows][NC];
#pragma unroll
        for (int r = 0; r < kRows; ++r)
#pragma unroll
            for (int n = 0; n < NC; ++n) acc[r][n] = 0.0f;
        if (active)
            decode_rows<NC, BPT, kRows>(smem + (size_t)slot * stage_bytes + row_off, rowbytes, abase,
                                        dbase, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        float vals[V];
#pragma unroll
        for (int i = 0; i < V; ++i) vals[i] = i < kRows * NC ? acc[i / NC][i % NC] : 0.0f;
        float total = warp_transpose_reduce<V>(vals, lane);
        const int row = c * SR + rg * kRows + vr;
        bool store = writer && row < nrows;
        if (WK > 1) {
            const int par = it & 1;
            float *rs = red + (size_t)(wid * 2 + par) * WK * kVMax;
            if (wk != 0) {
                if (it >= 2 && !mbar_wait(&redfree[wid * 2 + par], ((it >> 1) - 1) & 1)) {
                    record_status(a.status, RFP2_ETIMEOUT);
                    *abort_flag = 1;
                    return;
                }
                if (writer) rs[wk * kVMax + idx] = total;
                __syncwarp();
                if (lane == 0) mbar_arrive(&redfull[wid * 2 + par]);
                store = false;
            } else {
                if (!mbar_wait(&redfull[wid * 2 + par], (it >> 1) & 1)) {
                    record_status(a.status, RFP2_ETIMEOUT);
                    *abort_flag = 1;
                    return;
                }
                if (writer)
                    for (int j = 1; j < WK; ++j) total += rs[j * kVMax + idx];
                __syncwarp();
                if (lane == 0) mbar_arrive(&redfree[wid * 2 + par]);
            }
        }
        if (store) a.y[(int64_t)vn * a.M + r_begin + row] = total;
        next_slot();
    }
}

// ---------------------------------------------------------------------------
// Host side

struct Plan {
    int bpt, WK, H, stages, grid;
    size_t smem;
    uint32_t off_bars, off_red, off_actq, off_actd;
};

size_t align16(size_t v) { return (v + 15) / 16 * 16; }

int cw_for(int NC) { return NC <= 3 ? cw_of<1>() : cw_of<4>(); }

// K-slices of a row (a power of two) when each lane takes bpt blocks.
int k_slices(int64_t KB, int bpt) {
    const int64_t need = (KB + 32 * bpt - 1) / (32 * bpt);
    int w = 1;
    while (w < need) w *= 2;
    return w;
}

bool make_plan(int NC, int64_t M, int64_t K, bool fq, const void *x, Plan &p) {
    (void)fq;
    (void)x;
    const int kCW = cw_for(NC);
    if (K % 256 != 0 || K <= 0 || M <= 0) return false;
    const int64_t KB = K / 32;
    int bpt = 4;
    while (bpt > 1 && KB < 32 * bpt) bpt /= 2;
    int WK = k_slices(KB, bpt);
    if (WK > kCW) {
        bpt = 8;
        WK = k_slices(KB, bpt);
    }
    if (WK > kCW) return false;
    p.bpt = bpt;
    p.WK = WK;
    const int64_t rowbytes = KB * 10;
    const int sms = sm_count(current_device());
    const size_t actq = (size_t)NC * WK * bpt * 1024;
    const size_t actd = (size_t)NC * WK * bpt * 128;
    const size_t red = WK > 1 ? (size_t)kCW * 2 * kVMax * 4 : 0;
    // two sets of warps on alternate stages where a set still spans a row
    // and each set gets at least one ring slot; else one set
    for (int H = (NC == 1 && 2 * WK <= kCW) ? 2 : 1; H >= 1; --H) {
        const int G = kCW / H, RGS = G / WK, SR = kRows * RGS;
        const int64_t stage = (int64_t)SR * rowbytes;
        const int64_t stages_total = (M + SR - 1) / SR;
        p.H = H;
        p.grid = (int)(stages_total < sms ? stages_total : sms);
        const int64_t rows_per_cta = (M + p.grid - 1) / p.grid;
        const int64_t stages_per_cta = (rows_per_cta + SR - 1) / SR;
        for (int attempt = 0; attempt < 2; ++attempt) {
            const size_t budget = attempt == 0 ? kSmemPair : kSmemOne;
            int S = (int)std::min<int64_t>(stages_per_cta, kMaxStages);
            for (; S >= 1; --S) {
                const size_t bars = align16((size_t)(2 * S + 1 + 4 * kCW) * 8 + 4);
                if ((size_t)S * stage + actq + actd + red + bars <= budget) break;
            }
            if (S < 1 || (S < H && stages_per_cta > 1)) continue;
            p.stages = S;
            size_t off = (size_t)S * stage;
            p.off_actq = (uint32_t)off;
            off += actq;
            p.off_actd = (uint32_t)off;
            off += actd;
            p.off_red = (uint32_t)off;
            off += red;
            p.off_bars = (uint32_t)off;
            off += align16((size_t)(2 * S + 1 + 4 * kCW) * 8 + 4);
            p.smem = off;
            return true;
        }
    }
    return false;
}

template <int NC, int BPT, bool FQ>
cudaError_t launch_t(const Plan &p, GsArgs &a, cudaStream_t stream) {
    auto kern = gemv_stream_kernel<NC, BPT, FQ>;
    static std::mutex mu;
    static int configured[64] = {0};
    const int dev = current_device();
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && configured[dev] == 0) {
            cudaError_t e = set_smem_limit(kern, (int)kSmemOne);
            if (e != cudaSuccess) return e;
            configured[dev] = 1;
        }
    }
    return launch(kern, dim3(p.grid), dim3((cw_of<NC>() + 1) * 32), p.smem, stream, true, a);
}

template <int NC, bool FQ>
cudaError_t launch_nc(const Plan &p, GsArgs &a, cudaStream_t stream) {
    switch (p.bpt) {
        case 8: return launch_t<NC, 8, FQ>(p, a, stream);
        case 4: return launch_t<NC, 4, FQ>(p, a, stream);
        case 2: return launch_t<NC, 2, FQ>(p, a, stream);
        default: return launch_t<NC, 1, FQ>(p, a, stream);
    }
}

// One launch for N columns: the GEMV on pre-quantized q/d (x == nullptr) or
// quantizing x itself (q/d copies to qout/dout when given).
cudaError_t launch_cols(const uint8_t *W, int64_t M, int64_t K, const int8_t *q, const float *d,
                        const float *x, int64_t N, int8_t *qout, float *dout, float *y,
                        int32_t *status, cudaStream_t stream) {
    const bool fq = x != nullptr;
    Plan p;
    if (!make_plan((int)N, M, K, fq, x, p)) return cudaErrorInvalidValue;
    GsArgs a;
    a.W = W;
    a.q = q;
    a.d = d;
    a.x = x;
    a.qout = qout;
    a.dout = dout;
    a.y = y;
    a.status = status;
    a.M = (int)M;
    a.K = (int)K;
    a.WK = p.WK;
    a.H = p.H;
    a.stages = p.stages;
    a.rows_per_cta = (int)(M / p.grid);
    a.rows_extra = (int)(M % p.grid);
    a.x_vec = fq && aligned(x, 16) ? 1 : 0;
    // without the switch, W is read only after the earlier work completed
    a.w_early = weight_prefetch() ? 1 : 0;
    a.off_bars = p.off_bars;
    a.off_red = p.off_red;
    a.off_actq = p.off_actq;
    a.off_actd = p.off_actd;
    switch (N) {
#define RFP2_CASE(n)                                                                 \
    case n:                                                                          \
        return fq ? launch_nc<n, true>(p, a, stream) : launch_nc<n, false>(p, a, stream);
        RFP2_CASE(1)
        RFP2_CASE(2)
        RFP2_CASE(3)
        RFP2_CASE(4)
        RFP2_CASE(5)
        RFP2_CASE(6)
        RFP2_CASE(7)
        RFP2_CASE(8)
#undef RFP2_CASE
    }
    return cudaErrorInvalidValue;
}

// The GEMV for N columns.  The quantized activations of all columns live in
// shared memory; when they do not fit beside a weight ring (long rows at
// several columns), the columns go in groups of as many as fit, one launch
// each (every group streams W once).
cudaError_t launch_gemv(const uint8_t *W, int64_t M, int64_t K, const int8_t *q, const float *d,
                        const float *x, int64_t N, int8_t *qout, float *dout, float *y,
                        int32_t *status, cudaStream_t stream) {
    const bool fq = x != nullptr;
    Plan p;
    int64_t per = N;
    while (per > 1 && !make_plan((int)per, M, K, fq, x, p)) --per;
    const int64_t KB = K / 32;
    for (int64_t n0 = 0; n0 < N; n0 += per) {
        const int64_t nc = std::min(per, N - n0);
        const cudaError_t e = launch_cols(
            W, M, K, q ? q + n0 * K : nullptr, d ? d + n0 * KB : nullptr, x ? x + n0 * K : nullptr,
            nc, qout ? qout + n0 * K : nullptr, dout ? dout + n0 * KB : nullptr, y + n0 * M, status,
            stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

rfp2_status check_gemv_shape(int64_t M, int64_t K, int64_t N, bool fq, const void *x) {
    if (M <= 0 || K <= 0 || N < 1 || N > RFP2_MAX_BATCH) return RFP2_ESHAPE;
    if (M > (1LL << 30) || K > (1LL << 30)) return RFP2_ESHAPE;
    if (K % 256 != 0) return RFP2_EUNSUPPORTED;
    Plan p;  // one column always fits when any shape does
    if (!make_plan(1, M, K, fq, x, p)) return RFP2_EUNSUPPORTED;
    return RFP2_OK;
}

}  // namespace

size_t gemv_workspace_bytes(int64_t N, int64_t K) {
    const size_t qb = ((size_t)(N * K) + 255) / 256 * 256;
    return qb + (size_t)(N * (K / 32)) * sizeof(float);
}

}  // namespace rfp2

using namespace rfp2;

extern "C" rfp2_status rfp2_gemv_q8(const uint8_t *W, int64_t M, int64_t K, const int8_t *q,
                                    const float *d, int64_t N, float *y, int32_t *dev_status,
                                    rfp2_stream_t stream) {
    if (!W || !q || !d || !y) return RFP2_EINVAL;
    const rfp2_status st = check_gemv_shape(M, K, N, false, nullptr);
    if (st != RFP2_OK) return st;
    if (!aligned(W, 16) || !aligned(q, 16) || !aligned(d, 16) || !aligned(y, 4)) return RFP2_EALIGN;
    return from_cuda(launch_gemv(W, M, K, q, d, nullptr, N, nullptr, nullptr, y, dev_status,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" size_t rfp2_gemv_workspace_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0) return 0;
    return gemv_workspace_bytes(N, K);
}

extern "C" rfp2_status rfp2_gemv(const uint8_t *W, int64_t M, int64_t K, const float *x,
                                 int64_t N, float *y, void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, rfp2_stream_t stream) {
    if (!W || !x || !y) return RFP2_EINVAL;
    const rfp2_status st = check_gemv_shape(M, K, N, true, x);
    if (st != RFP2_OK) return st;
    if (!workspace || workspace_bytes < gemv_workspace_bytes(N, K)) return RFP2_EWORKSPACE;
    if (!aligned(W, 16) || !aligned(x, 4) || !aligned(y, 4) || !aligned(workspace, 256))
        return RFP2_EALIGN;
    int8_t *q = static_cast<int8_t *>(workspace);
    float *d = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                         ((size_t)(N * K) + 255) / 256 * 256);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Every CTA quantizes x itself (one launch): a separate quantize launch
    // and its dependency hop cost more than the redundant quantization, also
    // at eight columns (measured).
    if (N <= kFusedMaxN)
        return from_cuda(launch_gemv(W, M, K, nullptr, nullptr, x, N, q, d, y, dev_status, s));
    cudaError_t e = launch_quantize(x, N, K, q, d, s, true);
    if (e != cudaSuccess) return RFP2_ECUDA;
    return from_cuda(launch_gemv(W, M, K, q, d, nullptr, N, nullptr, nullptr, y, dev_status, s));
}

// ---------------------------------------------------------------------------
// rfp2_gemv_noalloc: rfp2_gemv for callers that cannot allocate device
// memory.  Some callers run where a cudaMalloc is not allowed or not
// possible: a plugin inside another runtime that owns the device memory
// pool, code running under a memory budget that must not grow, or a path that
// has to work after the pool is exhausted.  For them the quantized
// activations (the scratch the two-launch form of the GEMV passes from its
// quantize kernel to its GEMV kernel) live in a fixed array in device global
// memory that belongs to the library: every GPU that loads the library holds
// it until the process exits.  The array is shared by every call on a device,
// so calls that overlap on the GPU (different streams, different host
// threads) race on it and must be serialized by the caller.  Nothing in it
// needs to start at zero: each call overwrites the part it uses.

namespace rfp2 {
namespace {

// q int8 [N, K] (N*K <= kNoAllocMaxNK bytes) followed by d fp32 [N, K/32].
constexpr int64_t kNoAllocMaxNK = 65536;
constexpr size_t kNoAllocQBytes = kNoAllocMaxNK;
constexpr size_t kNoAllocBytes = kNoAllocQBytes + kNoAllocMaxNK / 32 * sizeof(float);
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];

// Device address of the array in the current context.  In host code the
// array's name is only a host-side stand-in; the address is looked up on
// every call (a host-side table lookup that allocates nothing), so a device
// reset or another context on the same device never leaves a stale address.
uint8_t *noalloc_scratch_ptr(cudaError_t *err) {
    void *p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    return *err == cudaSuccess ? static_cast<uint8_t *>(p) : nullptr;
}

}  // namespace
}  // namespace rfp2

extern "C" rfp2_status rfp2_gemv_noalloc(const uint8_t *W, int64_t M, int64_t K, const float *x,
                                         int64_t N, float *y, int32_t *dev_status,
                                         rfp2_stream_t stream) {
    if (!W || !x || !y) return RFP2_EINVAL;
    if (M <= 0 || K <= 0 || N < 1 || N > RFP2_MAX_BATCH) return RFP2_ESHAPE;
    if (N * K > kNoAllocMaxNK) return RFP2_EWORKSPACE;  // beyond the built-in scratch
    const rfp2_status st = check_gemv_shape(M, K, N, false, nullptr);
    if (st != RFP2_OK) return st;
    if (!aligned(W, 16) || !aligned(x, 4) || !aligned(y, 4)) return RFP2_EALIGN;
    cudaError_t e = cudaSuccess;
    uint8_t *scratch = noalloc_scratch_ptr(&e);
    if (!scratch) return RFP2_ECUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int8_t *q = reinterpret_cast<int8_t *>(scratch);
    float *d = reinterpret_cast<float *>(scratch + kNoAllocQBytes);
    // two launches: quantize into the scratch, then the GEMV reading it
    e = launch_quantize(x, N, K, q, d, s, true);
    if (e != cudaSuccess) return RFP2_ECUDA;
    return from_cuda(launch_gemv(W, M, K, q, d, nullptr, N, nullptr, nullptr, y, dev_status, s));
}
