// Dense ROCmFP2 GEMV: y[n, m] = sum_k w[m, k] * q[n, k] * dA (int8 path).
//
// Source: "ROCmFP2 codebook research report", sections "01 Storage",
// "02 Quantization" and "03 Runtime" (LOAD -> SPREAD -> PERMUTE -> DOT4 ->
// RESCALE, with each block expanded once for every activation column).
//
// GB300 design.  The packed weights (2.5 bits per weight) are the only large
// stream; the decode is bound by the integer pipe (about 50 cycles of one SM
// sub-partition per 32 blocks, see rfp2_decode.cuh); the activations of a
// call have to be read and quantized after the kernel before has completed.
//  * Persistent grid, one CTA per SM, two CTAs resident per SM: the next
//    call's CTA becomes resident as soon as this one starts
//    (griddepcontrol.launch_dependents at entry), so its weight stream can
//    overlap this call (when weight prefetch is enabled; see
//    rfp2_set_weight_prefetch) and its barriers are ready when this call ends.
//  * CTA i owns the contiguous rows [i*M/G, (i+1)*M/G).  A producer warp
//    streams them in stages of kRows*RG rows (kRows rows per row group of
//    consumer warps) with 1-D bulk async copies (L2 evict-first) into a ring of as many
//    stages as fit; the rows that do not fit are prefetched into L2 at entry.
//  * The activations are read once per CTA (one bulk copy of x), quantized
//    by the consumer warps (Q8_1-style, bit-exact) and written to shared
//    memory already permuted into the lane order of expand_half, one 16-byte
//    word group per lane and half-block, so the decode loop reads them with
//    conflict-free 16-byte loads and keeps no activation registers.
//  * Each consumer warp takes kRows rows of every stage (independent rows in
//    flight, one barrier wait per kRows rows), keeps the per-lane partial
//    sums of up to 16 rows x columns in registers and reduces them across the
//    warp once per round (a transposing butterfly), so no stage ends with a
//    shuffle chain and a store.
//  * Every wait is an mbarrier wait with a time limit; a timeout stores
//    RFP2_ETIMEOUT and the CTA winds down after its copies have landed.
//    Rows split over several warps along K are combined through a
//    double-buffered shared-memory slot guarded by mbarriers, never bar.sync.
#include <mutex>

#include <algorithm>

#include "common.cuh"
#include "gemv_core.cuh"
#include "quantize.cuh"

namespace rfp2 {
namespace {

// Launch shapes (two CTAs per SM; CW consumer warps + 1 producer warp, each
// consumer decoding R rows of every stage at once).  One column: 16 warps of
// at most 56 registers, so four warps per SM sub-partition hide each other's
// latencies.  From two columns the extra activation and accumulator
// registers would spill at 56, so 8 warps of up to 112 registers.
#ifndef RFP2_GEMV_WIDE_CW
#define RFP2_GEMV_WIDE_CW 8
#endif
#ifndef RFP2_GEMV_WIDE_R
#define RFP2_GEMV_WIDE_R 2
#endif
template <int NC>
constexpr int cw_of() {
    return NC == 1 ? 16 : RFP2_GEMV_WIDE_CW;
}
template <int NC>
constexpr int rows_of() {
    return NC == 1 ? 2 : RFP2_GEMV_WIDE_R;
}
// Partial sums (rows x columns) a lane keeps before a warp reduction.
constexpr int kVMax = 16;
// Shared memory per CTA: two CTAs per SM, or one when a shape needs more.
constexpr size_t kSmemPair = 113 * 1024;
constexpr size_t kSmemOne = 227 * 1024;
constexpr int kMaxStages = 32;
// Largest batch quantized inside the GEMV kernel by every CTA.
constexpr int64_t kFusedMaxN = 8;

// Rows of a warp per reduction round: a multiple of R with RR * NC <= 16.
template <int NC, int R>
constexpr int round_rows() {
    return R * (kVMax / (R * NC) > 0 ? kVMax / (R * NC) : 1);
}
// Activation groups (four blocks) a warp handles per pass: the K = 4096 case
// spread evenly over the consumer warps.
template <int NC, int CW>
constexpr int act_groups_per_pass() {
    return 32 * NC / CW < 1 ? 1 : 32 * NC / CW > 4 ? 4 : 32 * NC / CW;
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
    int M, K, WK, RG, stages, rows_per_cta, rows_extra, x_tma, w_early;
    uint32_t off_bars, off_red, off_actq, off_actd, off_x;
};

// ---------------------------------------------------------------------------
// Activations in shared memory.  Column n, block B of the row (the K-slice
// warp wk = B / (32*BPT), lane l = (B / BPT) % 32, b = B % BPT) is slot
// ((n*WK + wk)*BPT + b) of the dA array [slot][32 lanes] and slots 2*that + h
// of the word array [slot][32 positions][4 words]: the half's 16 int8 values
// in the lane order of expand_half (0 2 4 6 | 8 10 12 14 | 1 3 5 7 | 9 11 13
// 15), lane l of slot s at position l ^ (s & 7).  The XOR keeps the decode's
// loads of a slot conflict-free (the 32 lanes still fill one 512-byte row)
// and spreads the stores of eight slots of one lane over all 32 banks.
// dA is stored times 2^19 (see block_sum_2m19).

RFP2_DEV uint32_t act_word_offset(int slot, int lane) {
    return ((uint32_t)slot * 32 + (uint32_t)(lane ^ (slot & 7))) * 16;
}

// Store the 4 int8 codes `word` (values 4*l8 .. 4*l8+3 of a block, l8 = lane
// & 7) of the block handled by this lane's group of eight lanes: lanes 2j and
// 2j+1 swap their words and each writes one permuted word.  Every lane of the
// warp must call this (a shuffle).  A group beyond the last one stores
// nothing; a block beyond K (an idle lane's slot) stores zeros.
RFP2_DEV void store_permuted(uint8_t *actq, float *actd, uint32_t word, float dA, bool in_range,
                             bool valid, int slot_b, int lane_c, int lane) {
    const int l8 = lane & 7;
    const uint32_t partner = __shfl_xor_sync(0xffffffffu, word, 1);
    const uint32_t w = (l8 & 1) ? prmt(partner, word, 0x7531u) : prmt(word, partner, 0x6420u);
    if (!in_range) return;
    const int h = l8 >> 2, jp = (l8 >> 1) & 1;
    const int wi = (l8 & 1) ? 2 + jp : jp;
    const int slot = slot_b * 2 + h;
    *reinterpret_cast<uint32_t *>(actq + act_word_offset(slot, lane_c) + wi * 4) = valid ? w : 0u;
    if (l8 == 0) actd[(size_t)slot_b * 32 + lane_c] = valid ? dA * 0x1p19f : 0.0f;
}

// Work split of the activation pass: groups of four consecutive blocks of a
// column (the row padded to WK*32*BPT blocks, so idle lanes get zeros), one
// group per warp instruction, eight lanes per block and four values per lane:
// the 512 bytes of x a group reads are contiguous.
struct ActGroup {
    int n, slot_b, lane_c, B;
};
// WK and BPT are powers of two: log_wk = log2(WK), so a column has
// WK * BPT * 8 = 2^(log_wk + log2(BPT) + 3) groups.
template <int BPT>
RFP2_DEV ActGroup act_group(int g, int lane, int log_wk) {
    constexpr int LB = Log2<BPT>::v;
    ActGroup r;
    const int lpc = log_wk + LB + 3;
    r.n = g >> lpc;
    r.B = ((g & ((1 << lpc) - 1)) << 2) + (lane >> 3);
    const int wkq = r.B >> (5 + LB);
    r.lane_c = (r.B >> LB) & 31;
    r.slot_b = (((r.n << log_wk) + wkq) << LB) + (r.B & (BPT - 1));
    return r;
}

RFP2_DEV float rcp_approx_f(float v) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// Quantize the NC x K activations (from global x or the bulk-copied shared
// copy xs) into the permuted shared layout; CTA 0 also writes q and d in
// natural layout to qout/dout.  Same results as the quantize kernel (d = amax
// / 127 and q = roundf(a / d), IEEE divisions): q comes from z = a *
// rcp.approx(d), whose relative error is below 2^-22; the IEEE quotient
// fl(a/d) lies within 2^-24 of a/d, so both round to the same integer unless
// a/d is within about 2^-21 |z| of a half-integer; lanes whose z is within
// 2^-19 |z| of one (or is not finite) take the IEEE division and roundf
// instead.  Away from half-integers z + 1.5*2^23 rounds z to that integer and
// holds it in its low mantissa bits; |z| <= 127 (1 + 2^-22) needs no clamp.
template <int NC, int BPT, int QB, int CW>
RFP2_DEV void quantize_permuted(const float *__restrict__ xsrc, bool vec, int K, int WK, int w,
                                int lane, uint8_t *actq, float *actd, int8_t *gq, float *gd) {
    const int KB = K >> 5;
    const int ngroups = NC * WK * BPT * 8;
    const int log_wk = __ffs(WK) - 1;
    const int l8 = lane & 7;
    for (int g0 = w; g0 < ngroups; g0 += CW * QB) {
        float v[QB][4];
        ActGroup G[QB];
        bool ok[QB], in[QB];
#pragma unroll
        for (int j = 0; j < QB; ++j) {
            const int g = g0 + j * CW;
            in[j] = g < ngroups;
            G[j] = act_group<BPT>(in[j] ? g : 0, lane, log_wk);
            ok[j] = in[j] && G[j].B < KB;
            const float *src = xsrc + (int64_t)G[j].n * K + (int64_t)G[j].B * 32 + l8 * 4;
            if (!ok[j]) {
                v[j][0] = v[j][1] = v[j][2] = v[j][3] = 0.0f;
            } else if (vec) {
                const float4 t = *reinterpret_cast<const float4 *>(src);
                v[j][0] = t.x;
                v[j][1] = t.y;
                v[j][2] = t.z;
                v[j][3] = t.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) v[j][e] = src[e];
            }
        }
        float m[QB];
#pragma unroll
        for (int j = 0; j < QB; ++j)
            m[j] = fmaxf(fmaxf(fabsf(v[j][0]), fabsf(v[j][1])), fmaxf(fabsf(v[j][2]), fabsf(v[j][3])));
#pragma unroll
        for (int off = 4; off >= 1; off >>= 1)
#pragma unroll
            for (int j = 0; j < QB; ++j) m[j] = fmaxf(m[j], __shfl_xor_sync(0xffffffffu, m[j], off));
        float dd[QB];
        uint32_t word[QB];
        bool need = false;
#pragma unroll
        for (int j = 0; j < QB; ++j) {
            dd[j] = __fdiv_rn(m[j], 127.0f);
            const float rc = dd[j] != 0.0f ? rcp_approx_f(dd[j]) : 0.0f;
            uint32_t wq = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float z = v[j][e] * rc;
                const float zb = z + 12582912.0f;
                const float dist = fabsf(z - (zb - 12582912.0f));
                need |= !(fmaf(fabsf(z), 0x1p-19f, dist) < 0.5f - 0x1p-30f);
                wq |= ((uint32_t)(__float_as_int(zb) - 0x4B400000) & 0xFFu) << (8 * e);
            }
            word[j] = wq;
        }
        if (__any_sync(0xffffffffu, need) && need) {
#pragma unroll
            for (int j = 0; j < QB; ++j) {
                if (dd[j] == 0.0f) continue;
                uint32_t wq = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float qf = fminf(fmaxf(roundf(__fdiv_rn(v[j][e], dd[j])), -127.0f), 127.0f);
                    wq |= ((uint32_t)static_cast<int>(qf) & 0xFFu) << (8 * e);
                }
                word[j] = wq;
            }
        }
#pragma unroll
        for (int j = 0; j < QB; ++j) {
            store_permuted(actq, actd, word[j], dd[j], in[j], ok[j], G[j].slot_b, G[j].lane_c, lane);
            if (gq && ok[j]) {
                *reinterpret_cast<uint32_t *>(gq + (int64_t)G[j].n * K + (int64_t)G[j].B * 32 + l8 * 4) =
                    word[j];
                if (l8 == 0) gd[(int64_t)G[j].n * KB + G[j].B] = dd[j];
            }
        }
    }
}

// Pre-quantized q/d from global memory into the permuted shared layout.
template <int NC, int BPT, int QB, int CW>
RFP2_DEV void permute_quantized(const int8_t *__restrict__ q, const float *__restrict__ d, int K,
                                int WK, int w, int lane, uint8_t *actq, float *actd) {
    const int KB = K >> 5;
    const int ngroups = NC * WK * BPT * 8;
    const int log_wk = __ffs(WK) - 1;
    const int l8 = lane & 7;
    for (int g0 = w; g0 < ngroups; g0 += CW * QB) {
        uint32_t word[QB];
        float dv[QB];
        ActGroup G[QB];
        bool ok[QB], in[QB];
#pragma unroll
        for (int j = 0; j < QB; ++j) {
            const int g = g0 + j * CW;
            in[j] = g < ngroups;
            G[j] = act_group<BPT>(in[j] ? g : 0, lane, log_wk);
            ok[j] = in[j] && G[j].B < KB;
            word[j] = ok[j] ? __ldg(reinterpret_cast<const uint32_t *>(
                                  q + (int64_t)G[j].n * K + (int64_t)G[j].B * 32 + l8 * 4))
                            : 0u;
            dv[j] = ok[j] ? __ldg(d + (int64_t)G[j].n * KB + G[j].B) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < QB; ++j)
            store_permuted(actq, actd, word[j], dv[j], in[j], ok[j], G[j].slot_b, G[j].lane_c, lane);
    }
}

// ---------------------------------------------------------------------------
// Decode of R rows (of one stage, row_stride apart) against the activations:
// acc[r][n] += sum over the lane's BPT blocks of dA*(d0*S0 + d1*S1), each
// block's sum formed as (d0*S0 + d1*S1) * 2^-19 by block_sum_2m19 and
// multiplied by the stored dA * 2^19.  The R rows share every activation load.

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
RFP2_DEV void decode_rows(const uint8_t *p0, size_t row_stride, const uint8_t *actq,
                          const float *actd, int wk, int WK, int lane, float (&acc)[R][NC]) {
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
            const int slot_b = (n * WK + wk) * BPT + b;
            const uint4 q0 = *reinterpret_cast<const uint4 *>(actq + act_word_offset(2 * slot_b, lane));
            const uint4 q1 = *reinterpret_cast<const uint4 *>(actq + act_word_offset(2 * slot_b + 1, lane));
            const float dA = actd[(size_t)slot_b * 32 + lane];
            const uint32_t lo[4] = {q0.x, q0.y, q0.z, q0.w};
            const uint32_t hi[4] = {q1.x, q1.y, q1.z, q1.w};
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
    constexpr int kRows = rows_of<NC>();
    extern __shared__ __align__(128) uint8_t smem[];
    // let the next call's grid become resident at once (beside this CTA); it
    // touches x, y and the workspace only after this grid has completed
    pdl_launch_dependents();
    const int KB = a.K >> 5;
    const int rowbytes = KB * 10;
    const int S = a.stages, RG = a.RG, WK = a.WK;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + a.off_bars);
    uint64_t *empty = full + S;
    uint64_t *act_bar = empty + S;
    uint64_t *xbar = act_bar + 1;
    uint64_t *redfull = xbar + 1;      // [RG][2]
    uint64_t *redfree = redfull + 2 * RG;  // [RG][2]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(redfree + 2 * RG);
    float *red = reinterpret_cast<float *>(smem + a.off_red);  // [RG][2][WK][kVMax]
    uint8_t *actq = smem + a.off_actq;
    float *actd = reinterpret_cast<float *>(smem + a.off_actd);
    float *xs = reinterpret_cast<float *>(smem + a.off_x);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bx = blockIdx.x;
    const int64_t r_begin = (int64_t)bx * a.rows_per_cta + min(bx, a.rows_extra);
    const int nrows = a.rows_per_cta + (bx < a.rows_extra ? 1 : 0);
    // a stage holds kRows rows per row group (rows rg, RG + rg, ... of it)
    const int nchunks = (nrows + kRows * RG - 1) / (kRows * RG);
    const uint32_t chunk_bytes = (uint32_t)(kRows * RG) * rowbytes;
    const uint8_t *src = a.W + r_begin * rowbytes;

    auto issue = [&](int c, uint64_t pol) {
        const int s = c % S;
        const uint32_t bytes = (uint32_t)min(kRows * RG, nrows - c * kRows * RG) * rowbytes;
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s_stream(smem + (size_t)s * chunk_bytes, src + (size_t)c * chunk_bytes, bytes,
                        &full[s], pol);
    };

    if (threadIdx.x == kCW * 32) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        mbar_init(act_bar, kCW);
        mbar_init(xbar, 1);
        for (int i = 0; i < 2 * RG; ++i) {
            mbar_init(&redfull[i], WK > 1 ? WK - 1 : 1);
            mbar_init(&redfree[i], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
        // rows beyond the ring: into L2 now (always safe, L2 is coherent), so
        // their copies into the ring later are short
        for (int c = S; c < nchunks; ++c)
            bulk_prefetch_l2(src + (size_t)c * chunk_bytes,
                             (uint32_t)min(kRows * RG, nrows - c * kRows * RG) * rowbytes);
        if (a.w_early) {
            const uint64_t pol = policy_evict_first();
            for (int c = 0; c < nchunks && c < S; ++c) issue(c, pol);
        }
    }
    __syncthreads();

    if (warp == kCW) {
        // ---- producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            pdl_wait();  // the earlier work (x, and W unless prefetching) is complete
            if (FQ && a.x_tma) {
                const uint32_t xbytes = (uint32_t)NC * a.K * 4;
                mbar_arrive_expect_tx(xbar, xbytes);
                bulk_g2s(xs, a.x, xbytes, xbar);
            }
            int c = 0;
            if (a.w_early) {
                c = min(nchunks, S);
            } else {
                for (; c < nchunks && c < S; ++c) issue(c, pol);
            }
            for (; c < nchunks; ++c) {
                const int s = c % S;
                if (!mbar_wait_sleepy(&empty[s], ((c / S) - 1) & 1)) {
                    record_status(a.status, RFP2_ETIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                issue(c, pol);
            }
            // every copy in flight lands before the CTA may exit
            for (int i = max(0, c - S); i < c; ++i)
                if (!mbar_wait(&full[i % S], (i / S) & 1)) record_status(a.status, RFP2_ETIMEOUT);
        }
        return;
    }

    // ---- consumers
    const int wk = warp % WK, rg = warp / WK;
    const int kb0 = (wk * 32 + lane) * BPT;
    const bool active = kb0 < KB;
    pdl_wait();
    if constexpr (FQ) {
        constexpr int QB = act_groups_per_pass<NC, kCW>();
        if (a.x_tma) {
            if (!mbar_wait(xbar, 0)) {
                record_status(a.status, RFP2_ETIMEOUT);
                *abort_flag = 1;
                return;
            }
            quantize_permuted<NC, BPT, QB, kCW>(xs, true, a.K, WK, warp, lane, actq, actd,
                                           bx == 0 ? a.qout : nullptr, a.dout);
        } else {
            const bool vec = (reinterpret_cast<uintptr_t>(a.x) & 15) == 0;
            quantize_permuted<NC, BPT, QB, kCW>(a.x, vec, a.K, WK, warp, lane, actq, actd,
                                           bx == 0 ? a.qout : nullptr, a.dout);
        }
    } else {
        permute_quantized<NC, BPT, act_groups_per_pass<NC, kCW>(), kCW>(a.q, a.d, a.K, WK, warp, lane,
                                                                     actq, actd);
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

    constexpr int RR = round_rows<NC, kRows>();
    constexpr int V = NextPow2<RR * NC>::v;
    constexpr int L = Log2<V>::v;
    constexpr int CPR = RR / kRows;  // stages (kRows rows each) per round
    int round = 0;
    for (int c0 = 0; c0 < nchunks; c0 += CPR, ++round) {
        // partial sums of the round, oldest first after the shifts below
        float part[V];
#pragma unroll
        for (int i = 0; i < V; ++i) part[i] = 0.0f;
        const int npairs = min(CPR, nchunks - c0);
#pragma unroll 1
        for (int pi = 0; pi < npairs; ++pi) {
            const int c = c0 + pi;
            if (*abort_flag || !mbar_wait(&full[c % S], (c / S) & 1)) {
                record_status(a.status, RFP2_ETIMEOUT);
                *abort_flag = 1;
                return;
            }
            // a row past the CTA's last one still lies inside the stage: it is
            // computed from stale bytes and never stored
            const uint8_t *p0 = smem + (size_t)(c % S) * chunk_bytes + (size_t)rg * rowbytes +
                                (active ? (size_t)kb0 * 10 : 0);
            float acc[kRows][NC];
#pragma unroll
            for (int r = 0; r < kRows; ++r)
#pragma unroll
                for (int n = 0; n < NC; ++n) acc[r][n] = 0.0f;
            if (active)
                decode_rows<NC, BPT, kRows>(p0, (size_t)RG * rowbytes, actq, actd, wk, WK, lane, acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[c % S]);
            // shift in the stage's partials at the top
#pragma unroll
            for (int i = 0; i + kRows * NC < V; ++i) part[i] = part[i + kRows * NC];
#pragma unroll
            for (int r = 0; r < kRows; ++r)
#pragma unroll
                for (int n = 0; n < NC; ++n) part[V - kRows * NC + r * NC + n] = acc[r][n];
        }
        // partial index idx holds, counted from the bottom of the live part
        // (rel = idx - (V - kRows*NC*npairs)), stage c0 + rel / (kRows*NC),
        // its row (rel / NC) % kRows and column rel % NC
        float total = warp_transpose_reduce<V>(part, lane);
        const int idx = lane >> (5 - L);
        const bool writer = (lane & ((32 >> L) - 1)) == 0;
        const int rel = idx - (V - kRows * NC * npairs);
        const int pair = rel >= 0 ? rel / (kRows * NC) : 0;
        const int rr = rel >= 0 ? (rel / NC) % kRows : 0;
        const int n = rel >= 0 ? rel % NC : 0;
        const int64_t row = (int64_t)(c0 + pair) * kRows * RG + rr * RG + rg;
        const bool store = writer && rel >= 0 && row < nrows;
        if (WK > 1) {
            const int par = round & 1;
            float *slot = red + ((size_t)(rg * 2 + par) * WK) * kVMax;
            if (wk != 0) {
                if (round >= 2 && !mbar_wait(&redfree[rg * 2 + par], ((round >> 1) - 1) & 1)) {
                    record_status(a.status, RFP2_ETIMEOUT);
                    *abort_flag = 1;
                    return;
                }
                if (writer) slot[wk * kVMax + idx] = total;
                __syncwarp();
                if (lane == 0) mbar_arrive(&redfull[rg * 2 + par]);
                continue;
            }
            if (!mbar_wait(&redfull[rg * 2 + par], (round >> 1) & 1)) {
                record_status(a.status, RFP2_ETIMEOUT);
                *abort_flag = 1;
                return;
            }
            if (writer)
                for (int j = 1; j < WK; ++j) total += slot[j * kVMax + idx];
            __syncwarp();
            if (lane == 0) mbar_arrive(&redfree[rg * 2 + par]);
        }
        if (store) a.y[(int64_t)n * a.M + r_begin + row] = total;
    }
}

// ---------------------------------------------------------------------------
// Host side

struct Plan {
    int bpt, WK, RG, stages, grid, x_tma;
    size_t smem;
    uint32_t off_bars, off_red, off_actq, off_actd, off_x;
};

size_t align16(size_t v) { return (v + 15) / 16 * 16; }

int cw_for(int NC) { return NC == 1 ? cw_of<1>() : cw_of<2>(); }
int rows_for(int NC) { return NC == 1 ? rows_of<1>() : rows_of<2>(); }

bool make_plan(int NC, int64_t M, int64_t K, bool fq, const void *x, Plan &p) {
    const int kCW = cw_for(NC), kRows = rows_for(NC);
    if (K % 256 != 0 || K <= 0 || M <= 0) return false;
    const int64_t KB = K / 32;
    int bpt = 4;
    while (bpt > 1 && KB < 32 * bpt) bpt /= 2;
    if (KB > (int64_t)kCW * 32 * 4) bpt = 8;
    const int64_t wk_need = (KB + 32 * bpt - 1) / (32 * bpt);
    int WK = 0;
    for (int dv = 1; dv <= kCW; ++dv)
        if (kCW % dv == 0 && dv >= wk_need) {
            WK = dv;
            break;
        }
    if (WK == 0) return false;
    p.bpt = bpt;
    p.WK = WK;
    p.RG = kCW / WK;
    const int64_t rowbytes = KB * 10;
    const int64_t chunk = (int64_t)kRows * p.RG * rowbytes;
    const int sms = sm_count(current_device());
    const int64_t chunks_total = (M + kRows * p.RG - 1) / (kRows * p.RG);
    p.grid = (int)(chunks_total < sms ? chunks_total : sms);
    const int64_t rows_per_cta = (M + p.grid - 1) / p.grid;
    const int64_t chunks_per_cta = (rows_per_cta + kRows * p.RG - 1) / (kRows * p.RG);
    const size_t actq = (size_t)NC * WK * bpt * 1024;
    const size_t actd = (size_t)NC * WK * bpt * 128;
    const size_t xbytes = (size_t)NC * K * 4;
    for (int attempt = 0; attempt < 4; ++attempt) {
        const size_t budget = attempt < 2 ? kSmemPair : kSmemOne;
        const bool xt = fq && x && aligned(x, 16) && (attempt % 2 == 0);
        int S = (int)std::min<int64_t>(chunks_per_cta, kMaxStages);
        for (; S >= 1; --S) {
            size_t off = (size_t)S * chunk;
            const size_t bars = align16((size_t)(2 * S + 2 + 4 * p.RG + 1) * 8);
            const size_t red = WK > 1 ? (size_t)p.RG * 2 * WK * kVMax * 4 : 0;
            const size_t total = off + bars + red + actq + actd + (xt ? xbytes : 0);
            if (total <= budget) break;
        }
        if (S < 1) continue;
        p.stages = S;
        size_t off = (size_t)S * chunk;
        p.off_bars = (uint32_t)off;
        off += align16((size_t)(2 * S + 2 + 4 * p.RG + 1) * 8);
        p.off_red = (uint32_t)off;
        off += WK > 1 ? (size_t)p.RG * 2 * WK * kVMax * 4 : 0;
        p.off_actq = (uint32_t)off;
        off += actq;
        p.off_actd = (uint32_t)off;
        off += actd;
        p.off_x = (uint32_t)off;
        off += xt ? xbytes : 0;
        p.x_tma = xt ? 1 : 0;
        p.smem = off;
        return true;
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

// One launch: the GEMV on pre-quantized q/d (x == nullptr) or quantizing x
// itself (q/d copies to qout/dout when given).
cudaError_t launch_gemv(const uint8_t *W, int64_t M, int64_t K, const int8_t *q, const float *d,
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
    a.RG = p.RG;
    a.stages = p.stages;
    a.rows_per_cta = (int)(M / p.grid);
    a.rows_extra = (int)(M % p.grid);
    a.x_tma = p.x_tma;
    // without the switch, W is read only after the earlier work completed
    a.w_early = weight_prefetch() ? 1 : 0;
    a.off_bars = p.off_bars;
    a.off_red = p.off_red;
    a.off_actq = p.off_actq;
    a.off_actd = p.off_actd;
    a.off_x = p.off_x;
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

rfp2_status check_gemv_shape(int64_t M, int64_t K, int64_t N, bool fq, const void *x) {
    if (M <= 0 || K <= 0 || N < 1 || N > RFP2_MAX_BATCH) return RFP2_ESHAPE;
    if (M > (1LL << 30) || K > (1LL << 30)) return RFP2_ESHAPE;
    if (K % 256 != 0) return RFP2_EUNSUPPORTED;
    Plan p;
    if (!make_plan((int)N, M, K, fq, x, p)) return RFP2_EUNSUPPORTED;
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
