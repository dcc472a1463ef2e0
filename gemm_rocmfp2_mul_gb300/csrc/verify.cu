// ROCmFP2 GEMV for verify batches (tens to hundreds of tokens) on the
// 5th-generation tensor cores, with the results of the Q8_1 int path:
// y[n, m] = sum_b dA[n, b] * sum_{k in b} w[m, k] * q[n, k].
//
// Source: "ROCmFP2 codebook research report", section "03 Runtime" (Q8_1
// activations; expand each block once and reuse it for every activation
// column, the mid-range between the GEMV and the GEMM).
//
// Two launches chained with programmatic dependent launch:
//  1. vb_prep_kernel, one CTA per token: quantize it (Q8_1 blocks, the same
//     arithmetic as rfp2_gemv), then split x^ = q * dA scaled by 2^-kc into
//     two f16 pieces, hi + lo, relative residual <= 2^-22, written per tile
//     of BNT tokens as BNT hi rows then BNT lo rows, in the K order in which
//     the decode below lays out the weights (a fixed permutation inside
//     every 16 values);
//  2. vb_fused_kernel: one CTA per 128 weight rows x BNT tokens.
//     - warp 2 streams the packed blocks (128 rows x 8 blocks = 80 bytes a
//       row per stage) with 2-D TMA; it needs no earlier kernel, so it starts
//       before the dependency wait;
//     - sixteen decode warps (four groups of four, one TMEM lane quarter
//       each; group g takes every fourth 64-value slice, so each group has a
//       second slice of lookahead in the eight-slot ring) turn every block
//       into exact f16 levels * scale: per
//       half one byte table {-4s, -s, +s, +4s} (high bytes of the f16 values,
//       built from f16(s) with one byte add and one OR) and one PRMT per two
//       weights, the shared low byte coming from f16(s) itself; the 64-value
//       slices go straight into tensor memory (tcgen05.st), which the MMA
//       reads as its A operand: the decoded weights never touch shared
//       memory or HBM;
//     - warp 0 streams the activation tile (both pieces, one 2-D TMA box of
//       2*BNT rows, SWIZZLE_128B);
//     - warp 1 issues tcgen05.mma kind::f16 (A in TMEM, B in shared memory;
//       M = 128 weight rows, N = 2*BNT = the tokens' hi and lo pieces, K =
//       16, fp32 in TMEM); at BNT = 32 and 64 the k-steps alternate between
//       two accumulators, at BNT = 128 (65 tokens and up) one 256-column
//       accumulator takes them all.  The tensor cores' fp32 accumulation
//       does not round to nearest (over K = 4096 in one accumulator ~1.5e-5
//       relative), so no accumulator takes more than 128 MMAs before the
//       decode warps add it into fp32 registers (one weight row and a
//       quarter of the tokens per thread, hi + lo; every 64 stages with two
//       accumulators, 32 with one) and, at the end, store y with 2^kc.
#include <algorithm>
#include <mutex>

#include <cuda_fp16.h>

#include "common.cuh"
#include "rfp2_decode.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace rfp2 {
namespace {

constexpr int VBM = 128;                    // weight rows per tile (UMMA M, TMEM lanes)
constexpr int VSTEP = 64;                   // K per MMA stage (four UMMA k-steps of 16)
constexpr int VUK = 16;                     // K per UMMA instruction
constexpr int VPK = 256;                    // K per packed-weight stage (8 blocks)
constexpr int kPRowBytes = VPK / 32 * 10;   // 80 bytes of a row per packed stage
constexpr int kPStageBytes = VBM * kPRowBytes;
// Packed-weight stages in flight.
template <int BNT>
constexpr int vb_pstages() { return BNT <= 32 ? 8 : 3; }
constexpr int kMaxPStages = 8;
// TMEM: the accumulators (2 x 2*BNT fp32 columns, or 1 x 256 at BNT = 128),
// then the A ring of 32-column slots (64 f16 values of 128 rows) in what is
// left of the 512 columns: three steps of slots at BNT = 32, two at BNT = 64,
// three (of two stages) at BNT = 128.  The ring depth hides the
// tensor-memory store of a slot, which competes with the MMAs for tensor
// memory and waits for the MMAs that last read the slot.
// At BNT = 128 one accumulator (2*BNT = 256 columns) takes every k-step and
// the steps are two stages (an activation stage is 32 KB); below, two
// accumulators take alternate k-steps and the steps are four stages.
template <int BNT>
constexpr int vb_accs() { return BNT >= 128 ? 1 : 2; }
template <int BNT>
constexpr int vb_vq() { return BNT >= 128 ? 2 : 4; }  // MMA stages per step of the issuing warp
// MMA stages between two read-backs: at most 128 MMAs per accumulator
template <int BNT>
constexpr int vb_vround() { return 32 * vb_accs<BNT>(); }
template <int BNT>
constexpr int vb_bstages();
// A slots: what tensor memory leaves beside the accumulators, at most as many
// steps as the step barriers' ring holds (a slot is reused after the MMAs of
// the step that last read it, whose barrier must still be in the ring)
template <int BNT>
constexpr int vb_aslots() {
    return std::min((512 - vb_accs<BNT>() * 2 * BNT) / 32 / vb_vq<BNT>() * vb_vq<BNT>(),
                    vb_bstages<BNT>());
}
constexpr int kTmemCols = 512;
constexpr int kDecodeWarps = 16;
constexpr int kGroups = kDecodeWarps / 4;   // decode groups (one warp per TMEM lane quarter)
constexpr int VTHREADS = (4 + kDecodeWarps) * 32;  // 0 B loads, 1 MMA, 2 W loads, 3 idle, 4.. decode

// Activation stages (three steps of VQ).  The issuing warp works in steps of
// VQ stages with one ready barrier and one commit a step (an mbarrier probe
// costs ~100 cycles even on a completed phase, a commit ~140), and each
// step's activation tile arrives as one TMA box: the copy engine keeps few
// boxes in flight, so its throughput grows with the box.
template <int BNT>
constexpr int vb_bstages() { return 3 * vb_vq<BNT>(); }
// mbarriers (2 per activation stage, 2 per packed stage, 2 per A slot, 3
// more), the TMEM address and the abort flag
constexpr int kVbBarrierBytes = 1024;
static_assert((2 * 3 + 2 * kMaxPStages + 3) * 8 + 8 <= kVbBarrierBytes,
              "barrier region too small");
template <int BNT>
constexpr int vb_bstage_bytes() { return 2 * BNT * VSTEP * 2; }  // BNT hi rows, BNT lo rows
// at least 120 KB so that one CTA (and its 512 TMEM columns) owns the SM
template <int BNT>
constexpr size_t vb_smem_bytes() {
    return std::max<size_t>(1024 + (size_t)vb_bstages<BNT>() * vb_bstage_bytes<BNT>() +
                                (size_t)vb_pstages<BNT>() * kPStageBytes + kVbBarrierBytes,
                            120 * 1024);
}

// Position inside a 16-value group: MMA k-slot s holds the weight (and the
// activation) of index 4*(s % 4) + r(s / 4), r = (0, 2, 1, 3); the decode
// below produces the slots in this order.
__host__ __device__ constexpr int vb_slot_source(int s) {
    return 4 * (s & 3) + ((((s >> 2) & 1) << 1) | ((s >> 3) & 1));
}

// One CTA per token n (256 threads; thread i owns the 16-value groups
// g = i, i + 256, ...; a 32-value block is the group pair (2b, 2b + 1), held
// by neighbouring lanes).  Pass 1 quantizes: d = max|x| / 127 and q =
// round-half-away(x / d), both IEEE divisions, q and d stored to the
// workspace.  Then kc = ilogb(127 * max d) (every scaled value below 2) and
// pass 2 writes x^ = (q * d) * 2^-kc as two f16 pieces in MMA slot order.
__global__ void __launch_bounds__(256) vb_prep_kernel(const float *__restrict__ x, int K, int bnt,
                                                      int8_t *__restrict__ q,
                                                      float *__restrict__ d,
                                                      __half *__restrict__ xp, int *kc_out) {
    __shared__ float wmax[8];
    pdl_wait();
    pdl_launch_dependents();
    const int n = blockIdx.x, tid = threadIdx.x;
    const int G = K >> 4;  // 16-value groups (even: K % 32 == 0)
    const float *xr = x + (int64_t)n * K;
    int8_t *qr = q + (int64_t)n * K;
    float *dr = d + (int64_t)n * (K >> 5);
    float dmax = 0.0f;
    for (int base = 0; base < G; base += 256) {
        const int g = base + tid;
        const bool valid = g < G;  // G even and base even: pairs are both valid or both not
        float v[16];
        float amax = 0.0f;
        if (valid) {
            const float4 *src = reinterpret_cast<const float4 *>(xr + 16 * g);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 f = src[i];
                v[4 * i] = f.x;
                v[4 * i + 1] = f.y;
                v[4 * i + 2] = f.z;
                v[4 * i + 3] = f.w;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        if (valid) {
            const float dd = __fdiv_rn(amax, 127.0f);
            uint32_t packed[4] = {0u, 0u, 0u, 0u};
            if (dd != 0.0f) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float r = roundf(__fdiv_rn(v[i], dd));
                    r = fminf(fmaxf(r, -127.0f), 127.0f);
                    packed[i >> 2] |= ((uint32_t)(int)r & 0xFFu) << (8 * (i & 3));
                }
            }
            *reinterpret_cast<uint4 *>(qr + 16 * g) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            if ((g & 1) == 0) dr[g >> 1] = dd;
            dmax = fmaxf(dmax, dd);
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        dmax = fmaxf(dmax, __shfl_xor_sync(0xffffffffu, dmax, off));
    if ((tid & 31) == 0) wmax[tid >> 5] = dmax;
    __syncthreads();  // also publishes q and d to the whole CTA
    dmax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) dmax = fmaxf(dmax, wmax[i]);
    const float bound = 127.0f * dmax;  // >= max |q * dA| of the token
    const int kc = bound > 0.0f ? ilogbf(bound) : 0;
    if (tid == 0) kc_out[n] = kc;
    __half *xhi = xp + ((int64_t)(n / bnt) * 2 * bnt + n % bnt) * K;
    __half *xlo = xhi + (int64_t)bnt * K;
    for (int g = tid; g < G; g += 256) {
        const uint4 qw = *reinterpret_cast<const uint4 *>(qr + 16 * g);
        const uint32_t qv[4] = {qw.x, qw.y, qw.z, qw.w};
        const float dd = dr[g >> 1];
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            const int k = vb_slot_source(s);
            const int qk = (int)(int8_t)(qv[k >> 2] >> (8 * (k & 3)));
            const float val = ldexpf((float)qk * dd, -kc);
            const __half h = __float2half_rn(val);
            const __half l = __float2half_rn(val - __half2float(h));
            const uint32_t hb = __half_as_ushort(h), lb = __half_as_ushort(l);
            if (s & 1) {
                hi[s >> 1] |= hb << 16;
                lo[s >> 1] |= lb << 16;
            } else {
                hi[s >> 1] = hb;
                lo[s >> 1] = lb;
            }
        }
        uint4 *ho = reinterpret_cast<uint4 *>(xhi + 16 * g);
        uint4 *lo4 = reinterpret_cast<uint4 *>(xlo + 16 * g);
        ho[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        ho[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
        lo4[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        lo4[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
    }
}

// One 10-byte block -> 16 words of f16 pairs (two UMMA k-steps of 8 columns,
// half 0 then half 1), each weight = level * scale exactly.  The decode is
// bound by the integer pipe, so it is written to keep work off it:
//  * a UE4M3 scale byte read as E4M3 (sign clear) is 2s, so one cvt and two
//    packed multiplies give f16(s) and f16(4s) exactly (zero stays zero);
//  * per half, the high bytes of {-4s, -s, +s, +4s} come from one PRMT of
//    f16(s), f16(4s) and one OR of the sign bits; the low byte L is shared
//    by all four (the levels are powers of two) and comes from f16(s);
//  * a PRMT with selector nibbles (L, code, L, code') then writes two
//    finished f16 values; the selector shifts are multiplies (the FMA pipe).
RFP2_DEV uint32_t shl_fma(uint32_t x, uint32_t pow2) { return x * pow2; }
RFP2_DEV uint32_t shr_fma(uint32_t x, uint32_t pow2_32_minus) { return __umulhi(x, pow2_32_minus); }

RFP2_DEV void decode_block_f16(const Block &k, uint32_t *w) {
    uint32_t e2;  // E4M3 values of the two scale bytes: low half byte 0
    asm("{\n .reg .b16 sc;\n cvt.u16.u32 sc, %1;\n cvt.rn.f16x2.e4m3x2 %0, sc;\n}\n"
        : "=r"(e2)
        : "r"(k.scales));
    // UE4M3 has exponent bias 8: s = E4M3 / 2 and 4s = E4M3 * 2 (both exact)
    const __half2 e = *reinterpret_cast<const __half2 *>(&e2);
    const __half2 q1 = __hmul2(e, __float2half2_rn(0.5f));
    const __half2 q4 = __hmul2(e, __float2half2_rn(2.0f));
    const uint32_t h2 = *reinterpret_cast<const uint32_t *>(&q1);
    const uint32_t h4 = *reinterpret_cast<const uint32_t *>(&q4);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        // bytes for codes 0..3: hb(4s)|sign, hb(s)|sign, hb(s), hb(4s)
        const uint32_t t = __byte_perm(h2, h4, half ? 0x7337u : 0x5115u) | 0x00008080u;
        const uint32_t L = half ? 0x06060606u : 0x04040404u;  // byte 4 or 6: low byte of f16(s)
        const uint32_t c = half ? k.hi : k.lo;
        const uint32_t sa = (shl_fma(c, 16u) & 0x30303030u) | L;       // (c0, c4)  (c8, c12)
        const uint32_t sb = (c & 0x30303030u) | L;                      // (c2, c6)  (c10, c14)
        const uint32_t sc = (shl_fma(c, 4u) & 0x30303030u) | L;        // (c1, c5)  (c9, c13)
        const uint32_t sd = (shr_fma(c, 1u << 30) & 0x30303030u) | L;  // (c3, c7)  (c11, c15)
        uint32_t *o = w + 8 * half;
        o[0] = __byte_perm(t, h2, sa);
        o[1] = __byte_perm(t, h2, shr_fma(sa, 1u << 16));
        o[2] = __byte_perm(t, h2, sb);
        o[3] = __byte_perm(t, h2, shr_fma(sb, 1u << 16));
        o[4] = __byte_perm(t, h2, sc);
        o[5] = __byte_perm(t, h2, shr_fma(sc, 1u << 16));
        o[6] = __byte_perm(t, h2, sd);
        o[7] = __byte_perm(t, h2, shr_fma(sd, 1u << 16));
    }
}

template <int BNT>
__global__ void __launch_bounds__(VTHREADS, 1)
    vb_fused_kernel(const __grid_constant__ CUtensorMap pmap, const __grid_constant__ CUtensorMap xmap,
                    float *__restrict__ y, int Mw, int Ntok, int K, const int *__restrict__ kc,
                    int32_t *status) {
    constexpr int VQ = vb_vq<BNT>(), VROUND = vb_vround<BNT>(), NACC = vb_accs<BNT>();
    constexpr int SB = vb_bstages<BNT>();
    constexpr int BB = vb_bstage_bytes<BNT>();
    constexpr int QS = SB / VQ;  // step barriers
    constexpr int VPSTAGES = vb_pstages<BNT>();
    constexpr int kASlots = vb_aslots<BNT>();
    constexpr int kACol0 = NACC * 2 * BNT;
    constexpr int AQ = kASlots / VQ;  // steps of lookahead in the A ring
    static_assert(SB % VQ == 0 && kASlots % VQ == 0 && AQ >= 2 && QS >= 3, "step rings");
    static_assert(AQ <= QS, "A-slot lookahead within the ring of step barriers");
    static_assert(kACol0 + 32 * kASlots <= kTmemCols, "tensor memory");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *bring = smem;                       // [SB][hi | lo], 1024-aligned tiles
    uint8_t *pring = smem + (size_t)SB * BB;     // [VPSTAGES][128 rows][80 bytes]
    // fullq[u % QS]: the VQ stages of step u ready (activation tile landed,
    // A slots written); emptyq[u % QS]: step u's MMAs complete (its B stages
    // and A slots free again)
    uint64_t *fullq = reinterpret_cast<uint64_t *>(pring + (size_t)VPSTAGES * kPStageBytes);
    uint64_t *emptyq = fullq + QS;
    uint64_t *pfull = emptyq + QS;
    uint64_t *pempty = pfull + VPSTAGES;
    uint64_t *accf = pempty + VPSTAGES;  // a round of MMAs complete
    uint64_t *acce = accf + 1;          // the accumulators read back
    uint64_t *mdone = acce + 1;         // every MMA complete
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mdone + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile_m = blockIdx.x, tile_n = blockIdx.y;
    const int NT = K / VSTEP;   // MMA stages
    const int NP = K / VPK;     // packed-weight stages
    const int nrounds = (NT + VROUND - 1) / VROUND;
    constexpr int NB = 2 * BNT;   // MMA N: hi and lo pieces of BNT tokens

    if (threadIdx.x == 0) {
        prefetch_tensor_map(&pmap);
        prefetch_tensor_map(&xmap);
        for (int s = 0; s < QS; ++s) {
            // the TMA producer and the decode warps of the step's VQ stages
            mbar_init(&fullq[s], 1 + VQ * (kDecodeWarps / kGroups));
            mbar_init(&emptyq[s], 1);
        }
        for (int s = 0; s < VPSTAGES; ++s) {
            mbar_init(&pfull[s], 1);
            mbar_init(&pempty[s], kDecodeWarps);
        }
        mbar_init(accf, 1);
        mbar_init(acce, kDecodeWarps);
        mbar_init(mdone, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---- activation pieces (written by the split kernel): one box per step
            pdl_wait();
            const int NQ = NT / VQ;
            int u = 0;
            for (; u < NQ; ++u) {
                const int qs = u % QS;
                if (u >= QS && !mbar_wait(&emptyq[qs], ((u / QS) - 1) & 1)) {
                    record_status(status, RFP2_ETIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&fullq[qs], VQ * BB);
                tma_load_3d(bring + (size_t)qs * VQ * BB, &xmap, 0, tile_n * NB, u * VQ, &fullq[qs]);
            }
            // copies still in flight land before the CTA may exit
            for (int i = max(0, u - QS); i < u; ++i)
                if (!mbar_wait(&fullq[i % QS], (i / QS) & 1)) record_status(status, RFP2_ETIMEOUT);
        }
    } else if (warp == 2) {
        if (lane == 0) {
            // ---- packed weights: no earlier kernel writes them
            int p = 0;
            for (; p < NP; ++p) {
                const int s = p % VPSTAGES;
                if (p >= VPSTAGES && !mbar_wait(&pempty[s], ((p / VPSTAGES) - 1) & 1)) {
                    record_status(status, RFP2_ETIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                mbar_arrive_expect_tx(&pfull[s], kPStageBytes);
                tma_load_2d(pring + (size_t)s * kPStageBytes, &pmap, p * kPRowBytes, tile_m * VBM,
                            &pfull[s]);
            }
            for (int i = max(0, p - VPSTAGES); i < p; ++i)
                if (!mbar_wait(&pfull[i % VPSTAGES], (i / VPSTAGES) & 1))
                    record_status(status, RFP2_ETIMEOUT);
        }
    } else if (warp == 1) {
        // ---- MMA issuer (the whole warp; one elected lane issues): step u =
        // stages VQ*u .. VQ*u + VQ - 1; stage t reads A slot t % kASlots and
        // B stage t % SB; k-step kk goes to accumulator kk % NACC; round r =
        // stages [VROUND*r, VROUND*(r + 1)) starts the accumulators afresh
        // (32/64-token tiles: VQ 4, 12/8 A slots, rounds of 64 stages, two
        // accumulators; 128-token tiles: VQ 2, 6 A slots, rounds of 32
        // stages, one accumulator).  The next step's barrier probe is issued
        // before this step's MMAs; the abort flag is read every other step.
        constexpr uint32_t idesc = idesc_f16_f32(VBM, NB);
        const uint64_t bdesc0 = smem_desc_sw128(smem_addr(bring));
        const uint32_t a_tmem0 = tmem + (uint32_t)kACol0;
        const int NQ = NT / VQ;
        bool ready = NQ > 0 && mbar_try_wait(&fullq[0], 0);
        for (int u = 0; u < NQ; ++u) {
            const int qs = u % QS, r = (u * VQ) / VROUND;
            const bool fresh = (u * VQ) % VROUND == 0;
            bool bad = (u % 2 == 0) && *abort_flag;
            bad = bad || (fresh && r >= 1 && !mbar_wait(acce, (r - 1) & 1));
            bad = bad || (!ready && !mbar_wait(&fullq[qs], (u / QS) & 1));
            if (__any_sync(0xffffffffu, bad)) {  // the lanes leave together
                if (lane == 0) record_status(status, RFP2_ETIMEOUT);
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            ready = u + 1 < NQ && mbar_try_wait(&fullq[(u + 1) % QS], ((u + 1) / QS) & 1);
            if (elect_one()) {
#pragma unroll
                for (int st = 0; st < VQ; ++st) {
                    const int t = u * VQ + st;
                    const uint32_t a_tmem = a_tmem0 + (uint32_t)((t % kASlots) * 32);
                    const uint64_t bdesc = bdesc0 + (uint64_t)(((t % SB) * BB) >> 4);
#pragma unroll
                    for (int kk = 0; kk < VSTEP / VUK; ++kk)
                        umma_f16_tmem_a(tmem + (uint32_t)((kk % NACC) * NB), a_tmem + 8 * kk,
                                        bdesc + 2 * kk, idesc,
                                        (fresh && st == 0 && kk < NACC) ? 0u : 1u);
                }
                umma_commit(&emptyq[qs]);  // frees the step's B stages and A slots
                if (((u + 1) * VQ) % VROUND == 0 || u == NQ - 1) umma_commit(accf);
            }
            __syncwarp();
        }
        if (elect_one()) umma_commit(mdone);
        __syncwarp();
        if (!mbar_wait(mdone, 0) && lane == 0) record_status(status, RFP2_ETIMEOUT);
    } else if (warp >= 4) {
        // ---- decode: group g takes slice g of every packed stage (stage t =
        // 4p + g), then reads back its quarter of the tokens
        const int g = (warp - 4) >> 2, q = warp & 3;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const uint8_t *prow = pring + (size_t)(32 * q + lane) * kPRowBytes + 20 * g;
        constexpr int TQ = BNT / kGroups;  // tokens read back by this thread
        float acc[TQ];
#pragma unroll
        for (int i = 0; i < TQ; ++i) acc[i] = 0.0f;
        bool ok = true;
        int drained = 0;  // rounds read back so far
        auto drain = [&](int r) {
            if (*abort_flag || !mbar_wait(accf, r & 1)) {
                record_status(status, RFP2_ETIMEOUT);
                *abort_flag = 1;
                return false;
            }
            tc_fence_after();
            constexpr int TC = TQ < 16 ? TQ : 16;  // columns per read
#pragma unroll
            for (int j = 0; j < NACC; ++j)
#pragma unroll
                for (int piece = 0; piece < 2; ++piece)
#pragma unroll
                    for (int c0 = 0; c0 < TQ; c0 += TC) {
                        uint32_t v[TC];
                        tmem_ld_cols<TC>(lane_base + tmem +
                                             (uint32_t)(j * NB + piece * BNT + g * TQ + c0),
                                         v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < TC; ++i) acc[c0 + i] += __uint_as_float(v[i]);
                    }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce);
            return true;
        };
        for (int t = g; t < NT && ok; t += kGroups) {
            // entering round r + 1: read back round r first (its MMAs need
            // nothing more from this group; the next round's wait for it)
            if (t >= (drained + 1) * VROUND) {
                if (!drain(drained)) { ok = false; break; }
                ++drained;
            }
            const int p = t / 4, ps = p % VPSTAGES, as = t % kASlots;
            if (*abort_flag || !mbar_wait(&pfull[ps], (p / VPSTAGES) & 1)) {
                record_status(status, RFP2_ETIMEOUT);
                *abort_flag = 1;
                break;
            }
            // this slice's 20 bytes of the row: blocks 2g and 2g + 1 of the stage
            const uint32_t *src = reinterpret_cast<const uint32_t *>(prow + (size_t)ps * kPStageBytes);
            uint32_t v[5];
#pragma unroll
            for (int i = 0; i < 5; ++i) v[i] = src[i];
            __syncwarp();
            if (lane == 0) mbar_arrive(&pempty[ps]);
            // decode first (overlapping the MMAs still reading the slot),
            // then wait for slot as, last read by MMA stage t - kASlots (step u - AQ)
            uint32_t w[32];
            decode_block_f16(block_from_words<2>(v, 0), w);
            decode_block_f16(block_from_words<2>(v, 1), w + 16);
            const int u = t / VQ;
            if (u >= AQ && (*abort_flag || !mbar_wait(&emptyq[(u - AQ) % QS], ((u - AQ) / QS) & 1))) {
                record_status(status, RFP2_ETIMEOUT);
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            tmem_st_32cols(tmem + lane_base + (uint32_t)(kACol0 + as * 32), w);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&fullq[u % QS]);
        }
        if (ok && !*abort_flag) {
            while (drained < nrounds && drain(drained)) ++drained;
        }
        pdl_wait();  // kc comes from the split kernel
        const int m = tile_m * VBM + q * 32 + lane;
        if (drained == nrounds && m < Mw) {
#pragma unroll
            for (int i = 0; i < TQ; ++i) {
                const int n = tile_n * BNT + g * TQ + i;
                if (n < Ntok) y[(int64_t)n * Mw + m] = acc[i] * ldexpf(1.0f, kc[n]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

struct VbWs {
    int8_t *q;
    float *d;
    __half *xp;  // [tiles][hi | lo][BNT][K]
    int *kc;
    size_t bytes;
};

int64_t vb_bnt(int64_t N) { return N <= 32 ? 32 : N <= 64 ? 64 : 128; }
int64_t vb_tiles_n(int64_t N) { return (N + vb_bnt(N) - 1) / vb_bnt(N); }

VbWs carve_vb(void *ws, int64_t M, int64_t K, int64_t N) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    uint8_t *p = static_cast<uint8_t *>(ws);
    VbWs w;
    size_t o = 0;
    w.q = reinterpret_cast<int8_t *>(p + o);
    o += up((size_t)N * K);
    w.d = reinterpret_cast<float *>(p + o);
    o += up((size_t)N * (K / 32) * 4);
    w.xp = reinterpret_cast<__half *>(p + o);
    o += up((size_t)vb_tiles_n(N) * 2 * vb_bnt(N) * K * 2);
    w.kc = reinterpret_cast<int *>(p + o);
    o += up((size_t)N * 4);
    w.bytes = o;
    return w;
}

template <int BNT>
cudaError_t launch_vb_fused(const uint8_t *W, const VbWs &w, float *y, int64_t M, int64_t K,
                            int64_t N, int32_t *status, cudaStream_t s) {
    CUtensorMap pmap, xmap;
    const uint64_t row_bytes = (uint64_t)(K / 32) * 10;
    const uint64_t xrows = (uint64_t)vb_tiles_n(N) * 2 * BNT;
    // activations as [K/64 slices][rows][64 values]: one box = VQ slices of
    // the tile's 2*BNT rows, laid out as VQ consecutive SWIZZLE_128B tiles
    const uint64_t xdims[3] = {(uint64_t)VSTEP, xrows, (uint64_t)(K / VSTEP)};
    const uint64_t xstrides[2] = {(uint64_t)K * 2, (uint64_t)VSTEP * 2};
    const uint32_t xbox[3] = {(uint32_t)VSTEP, (uint32_t)(2 * BNT), (uint32_t)vb_vq<BNT>()};
    if (!encode_tensor_map_2d(&pmap, W, CU_TENSOR_MAP_DATA_TYPE_UINT8, row_bytes, (uint64_t)M,
                              row_bytes, kPRowBytes, VBM) ||
        !encode_tensor_map_3d(&xmap, w.xp, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xdims, xstrides, xbox,
                              CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    static std::mutex mu;
    static int configured[64] = {0};
    const int dev = current_device();
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && !configured[dev]) {
            cudaError_t e = set_smem_limit(vb_fused_kernel<BNT>, (int)vb_smem_bytes<BNT>());
            if (e != cudaSuccess) return e;
            configured[dev] = 1;
        }
    }
    const dim3 grid((unsigned)((M + VBM - 1) / VBM), (unsigned)((N + BNT - 1) / BNT));
    return launch(vb_fused_kernel<BNT>, grid, dim3(VTHREADS), vb_smem_bytes<BNT>(), s, true, pmap,
                  xmap, y, (int)M, (int)N, (int)K, static_cast<const int *>(w.kc), status);
}

}  // namespace
}  // namespace rfp2

using namespace rfp2;

extern "C" size_t rfp2_gemv_batched_workspace_bytes(int64_t M, int64_t K, int64_t N) {
    if (M <= 0 || K <= 0 || N <= 0) return 0;
    return carve_vb(nullptr, M, K, N).bytes;
}

extern "C" rfp2_status rfp2_gemv_batched(const uint8_t *W, int64_t M, int64_t K, const float *x,
                                         int64_t N, float *y, void *workspace,
                                         size_t workspace_bytes, int32_t *dev_status,
                                         rfp2_stream_t stream) {
    if (!W || !x || !y) return RFP2_EINVAL;
    if (M <= 0 || K <= 0 || N <= 0) return RFP2_ESHAPE;
    if (M > (1LL << 30) || N > 65535 || K > (1 << 20)) return RFP2_ESHAPE;
    if (K % 256 != 0 || M % 16 != 0) return RFP2_EUNSUPPORTED;
    const VbWs w = carve_vb(workspace, M, K, N);
    if (!workspace || workspace_bytes < w.bytes) return RFP2_EWORKSPACE;
    if (!aligned(W, 16) || !aligned(x, 16) || !aligned(y, 4) || !aligned(workspace, 256))
        return RFP2_EALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch(vb_prep_kernel, dim3((unsigned)N), dim3(256), 0, s, true, x, (int)K,
                           (int)vb_bnt(N), w.q, w.d, w.xp, w.kc);
    if (e != cudaSuccess) return RFP2_ECUDA;
    if (N <= 32) e = launch_vb_fused<32>(W, w, y, M, K, N, dev_status, s);
    else if (N <= 64) e = launch_vb_fused<64>(W, w, y, M, K, N, dev_status, s);
    else e = launch_vb_fused<128>(W, w, y, M, K, N, dev_status, s);
    return from_cuda(e);
}
