// Prefill GEMM on the 5th-generation tensor cores:
// Y[n, m] = sum_k X[n, k] * w[m, k], X bf16 [N, K] (tokens), w the ROCmFP2
// weights [M, K] expanded exactly to bf16, Y fp32 [N, M].
//
// Source: "ROCmFP2 codebook research report", sections "02 Quantization"
// (weight = codebook[code] * UE4M3 scale: at most 4 significant bits times a
// power of two, hence exact in bf16) and "04 Measured evidence" (the
// end-to-end gain of the format comes from prefill, a dense contraction).
//
// rfp2_gemm is one launch: the GEMM decodes the packed blocks itself (warps
// 6-22 below); hfp4_gemm runs two:
//  1. expand: HFP4G32 rows -> bf16 rows in the workspace (one thread per
//     32-weight block, E2M1 x 2^(e-127), 64 bytes written per block); the f16
//     row scale is left to the GEMM's epilogue.
//  2. gemm: persistent over CTA pairs (clusters of two SMs), each pair walking
//     256-token x 256-weight-row tiles.  In each CTA warp 0 loads its 128
//     tokens and its 128 of the tile's weight rows, K-major 64-element slices
//     with 2-D TMA (SWIZZLE_128B) into a 6-stage ring (5 when decoding: the
//     ROCmFP2 boxes, 128 rows x 80 bytes = 256 K, stream into a 4-slot ring
//     and 16 decode warps write each K slice of B as exact bf16 in the same
//     swizzled layout, one weight row per thread); one thread of the even
//     CTA issues tcgen05.mma.cta_group::2 kind::f16 (M=256, N=256, K=16, bf16
//     in, fp32 accumulate) over both CTAs' stages, so each SM stores and reads
//     only half of the B operand; its commits free the stages of both CTAs and
//     signal both epilogues.  Warps 2-5 of each CTA read that CTA's 128 rows
//     of the accumulator back with tcgen05.ld and store fp32 rows while the
//     next tile's MMAs run in the other of two 256-column accumulators.  When
//     the last wave of whole tiles would leave most pairs idle, its tiles run
//     as 256 x 128 halves or 256 x 64 quarters spread over more pairs,
//     whichever ends the wave sooner.  Every wait is bounded; tensor memory
//     is always freed.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "expand.cuh"
#include "rfp2_decode.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace rfp2 {
namespace {

constexpr int BM = 128;  // tokens per CTA (TMEM lanes)
constexpr int PM = 256;  // tokens per CTA pair (UMMA M)
constexpr int BN = 256;  // weight rows per tile (UMMA N), half of them loaded by each CTA
constexpr int BK = 64;   // K per stage: one 128-byte swizzle row
constexpr int UK = 16;   // K per UMMA instruction
constexpr int kABytes = BM * BK * 2;
constexpr int kBBytes = (BN / 2) * BK * 2;  // this CTA's half of the B operand
constexpr int kStageBytes = kABytes + kBBytes;
constexpr uint32_t kTmemCols = 512;  // two 256-column accumulators
constexpr int kStgStride = 36;  // floats per row of an epilogue warp's 32 x 32 staging tile
constexpr int kStgFloats = 32 * kStgStride;
constexpr int BNH = BN / 2;  // weight rows of a half tile
// Packed ROCmFP2 weights decoded inside the GEMM: 128 rows x 80 bytes (eight
// 10-byte blocks = 256 K) per TMA box, one box per four K slices.
constexpr int kPBoxRowBytes = 80;
constexpr int kPBoxBytes = (BN / 2) * kPBoxRowBytes;
constexpr int kDecodeGroups = 4;         // group i decodes K slices i, i+4, ... (one per box)
constexpr int kDecodeGroupWarps = 4;     // 128 B rows per slice: one per thread
constexpr int kDecodeWarps = kDecodeGroups * kDecodeGroupWarps;

// Per B source: bf16 weights by TMA (kDecode false), or packed ROCmFP2 blocks
// decoded by kDecodeWarps warps into the B stages (kDecode true).
template <bool kDecode>
struct GemmCfg {
    static constexpr int kStages = kDecode ? 5 : 6;
    static constexpr int kPStages = kDecode ? 4 : 0;
    // warps: 0 A (and B) loads, 1 MMA, 2-5 epilogue; kDecode: 6 packed-box
    // loads, 7.. decode
    static constexpr int kThreads = (6 + (kDecode ? 1 + kDecodeWarps : 0)) * 32;
    static constexpr size_t kPRingOff = (size_t)kStages * kStageBytes;
    static constexpr size_t kBarOff = kPRingOff + (size_t)kPStages * kPBoxBytes;
    static constexpr size_t kStgOff = kBarOff + 256;
    static constexpr size_t kSmemBytes = 1024 + kStgOff + 4 * kStgFloats * 4;
};

// ---- expand ----------------------------------------------------------------
// OCP E2M1 code -> float: magnitude index k = c & 7 is 0 (0), 1 (0.5) or,
// for k >= 2, 2^((k >> 1) - 1) * (1 + (k & 1) / 2); bit 3 is the sign.
__device__ __forceinline__ float e2m1_float(uint32_t c) {
    const uint32_t k = c & 7;
    const uint32_t mag = k >= 2 ? ((((k >> 1) + 126) << 23) | ((k & 1) << 22)) : (k ? 0x3F000000u : 0u);
    return __uint_as_float(mag | ((c & 8) << 28));
}

// HFP4G32 rows -> bf16: element = E2M1[c] * 2^(e-127) (at most two
// significant bits times a power of two: exact in bf16, including the
// subnormal range; block byte 0xFF gives NaN), and the row scale row_scale_a
// (f16) as fp32, applied by the GEMM's epilogue.  One thread per 32-weight
// block; HFP4 "Element format (OCP E2M1)", "Block scale - UE8M0",
// "Per-row second-level scale (FP16)", "Byte layout - HFP4G32".
__global__ void __launch_bounds__(256) hfp4_expand_bf16_kernel(const uint8_t *__restrict__ W,
                                                               int M, int KB, int rb,
                                                               __nv_bfloat16 *__restrict__ out,
                                                               float *__restrict__ rs32) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= (int64_t)M * KB) return;
    const int64_t m = j / KB;
    const int b = (int)(j - m * KB);
    const uint8_t *row = W + m * rb;
    if (b == 0) rs32[m] = __half2float(__ushort_as_half((unsigned short)(row[0] | (row[1] << 8))));
    // the 17-byte block lies inside five aligned words (rows are 4-byte
    // aligned because K % 256 == 0): byte t of the block is byte t of u
    const uintptr_t addr = reinterpret_cast<uintptr_t>(row + 16 + 17 * b);
    const uint32_t *wp = reinterpret_cast<const uint32_t *>(addr & ~uintptr_t(3));
    const uint32_t sh = (uint32_t)(addr & 3) * 8;
    uint32_t v[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) v[i] = __ldg(wp + i);
    uint32_t u[5];
#pragma unroll
    for (int i = 0; i < 4; ++i) u[i] = __funnelshift_r(v[i], v[i + 1], sh);
    u[4] = v[4] >> sh;
    const uint32_t e = u[0] & 0xFFu;
    const float sc = __uint_as_float(e == 0 ? 0x00400000u : e == 0xFF ? 0x7FC00000u : e << 23);
    uint4 *o = reinterpret_cast<uint4 *>(out + j * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // 8 weights (code bytes 1+4q .. 4+4q) per 16-byte store
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = 1 + 4 * q + i;  // byte of the block
            const uint32_t byte = (u[t >> 2] >> (8 * (t & 3))) & 0xFFu;
            const float f0 = e2m1_float(byte & 15) * sc;
            const float f1 = e2m1_float(byte >> 4) * sc;
            w[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f0)) |
                   ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f1)) << 16);
        }
        o[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// ---- GEMM --------------------------------------------------------------------
// Schedule slot t -> output tile of a CTA pair.  Slots below t_full are whole
// 256-token x 256-weight-row tiles (token tile f % ntm of weight tile f / ntm,
// f = t); each tile after them takes 2^split_lg slots, one per part of its
// weight rows (256 >> split_lg of them).
struct Slot {
    int tile_m, col0;  // token tile of the pair; first weight row (output column)
    int width;         // weight rows (MMA N): 256, 128 or 64
};
__device__ __forceinline__ Slot slot_tile(int t, int t_full, int split_lg, int ntm) {
    if (t < t_full) return Slot{t % ntm, (t / ntm) * BN, BN};
    const int h = t - t_full, f = t_full + (h >> split_lg), w = BN >> split_lg;
    return Slot{f % ntm, (f / ntm) * BN + (h & ((1 << split_lg) - 1)) * w, w};
}

// Persistent over CTA pairs (clusters of two): pair p takes slots p, p + P,
// p + 2P, ...  CTA r of the pair loads tokens [256 tm + 128 r, +128) and
// weight rows [col0 + r n/2, +n/2) of each K slice into its own ring; the even
// CTA's MMA thread issues M = 256, N = n (256, or 128 / 64 for the parts of a
// split tile) pair MMAs over both CTAs' stages, so each SM reads and stores only its half of
// the B operand.  D rows of CTA r's tokens land in CTA r's tensor memory,
// alternating between two 256-column accumulators so the epilogue of one tile
// overlaps the MMAs of the next.  Barriers: full[s] (even CTA; both CTAs'
// copies complete on it), empty[s] and accf[b] (both CTAs; pair commits
// arrive on both), acce[b] (even CTA; the eight epilogue warps of the pair).
// colscale[m]: optional per-weight-row factor applied to every output.
//
// B maps: 128-, 64- and 32-row boxes for whole, half and quarter tiles.
// kDecode: wmap maps the packed ROCmFP2 weights (bytes, box 80 x 128 rows)
// and the other two are unused; warp 6 streams those boxes into a 4-slot
// ring, up to four boxes ahead of the decode, and warps 7-22 (four groups of
// four, group i taking K slice i of every box, one weight row of this CTA's
// B half per thread) decode each slice exactly to bf16, store it in the
// SWIZZLE_128B layout the TMA would have written, and arrive on the even
// CTA's full barrier.
template <bool kDecode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GemmCfg<kDecode>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                const __grid_constant__ CUtensorMap wmap_h, const __grid_constant__ CUtensorMap wmap_q,
                float *__restrict__ Y, int Ntok, int Mw, int K, int t_full, int split_lg,
                const float *__restrict__ colscale, int32_t *status) {
    using Cfg = GemmCfg<kDecode>;
    constexpr int kStages = Cfg::kStages, kPStages = Cfg::kPStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *pring = smem + Cfg::kPRingOff;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::kBarOff);
    uint64_t *empty = full + kStages;
    uint64_t *accf = empty + kStages;  // [2] accumulator b complete
    uint64_t *acce = accf + 2;         // [2] accumulator b read back (even CTA)
    uint64_t *pfull = acce + 2;        // [kPStages] packed box landed
    uint64_t *pempty = pfull + kPStages;  // [kPStages] packed box decoded
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(pempty + kPStages);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int nk = K / BK;
    const int ntm = (Ntok + PM - 1) / PM, ntn = (Mw + BN - 1) / BN;
    const int ntiles = ntm * ntn;
    const int nslots = t_full + ((ntiles - t_full) << split_lg);

    if (threadIdx.x == 0) {
        prefetch_tensor_map(&xmap);
        prefetch_tensor_map(&wmap);
        prefetch_tensor_map(&wmap_h);
        prefetch_tensor_map(&wmap_q);
        for (int s = 0; s < kStages; ++s) {
            // the producer's arrival (+ every decode warp of the pair)
            mbar_init(&full[s], kDecode ? 1 + 2 * kDecodeGroupWarps : 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 8);  // one arrival per epilogue warp of the pair
        }
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(&pfull[s], 1);
            mbar_init(&pempty[s], kDecodeWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync();  // barriers of both CTAs initialised before either signals the other
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    int g = 0;  // k-blocks loaded by this CTA (producer thread)
    if (warp == 0 && lane == 0) {
        // ---- TMA producer (both CTAs)
        pdl_wait();  // X (and the expanded weights) may come from earlier kernels
        const uint32_t full0 = cluster_map(&full[0], 0);
        for (int t = pair; t < nslots && !*abort_flag; t += npairs) {
            const Slot sl = slot_tile(t, t_full, split_lg, ntm);
            const int brows = sl.width / 2;
            const int arow = sl.tile_m * PM + (int)rank * BM, brow = sl.col0 + (int)rank * brows;
            for (int kb = 0; kb < nk; ++kb, ++g) {
                const int s = g % kStages;
                if (g >= kStages && !mbar_wait(&empty[s], ((g / kStages) - 1) & 1)) {
                    record_status(status, RFP2_ETIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                uint8_t *a = smem + (size_t)s * kStageBytes;
                if (kDecode) {
                    if (rank == 0) mbar_arrive_expect_tx(&full[s], 2u * (uint32_t)kABytes);
                    tma_load_2d_pair(a, &xmap, kb * BK, arow, full0 + 8u * s);
                } else {
                    if (rank == 0)
                        mbar_arrive_expect_tx(&full[s], 2u * (uint32_t)(kABytes + brows * BK * 2));
                    tma_load_2d_pair(a, &xmap, kb * BK, arow, full0 + 8u * s);
                    const CUtensorMap *bm = sl.width == BN ? &wmap : sl.width == BNH ? &wmap_h : &wmap_q;
                    tma_load_2d_pair(a + kABytes, bm, kb * BK, brow, full0 + 8u * s);
                }
            }
        }
    } else if (warp == 1 && rank == 0 && lane == 0) {
        // ---- MMA issuer (even CTA)
        int gm = 0, it = 0;
        bool ok = true;
        for (int t = pair; t < nslots && ok; t += npairs, ++it) {
            const int b = it & 1;
            if (it >= 2 && (*abort_flag || !mbar_wait(&acce[b], ((it >> 1) - 1) & 1))) {
                record_status(status, RFP2_ETIMEOUT);
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const uint32_t idesc = idesc_bf16_f32(PM, slot_tile(t, t_full, split_lg, ntm).width);
            const uint32_t d_tmem = tmem + (uint32_t)(b * BN);
            for (int kb = 0; kb < nk; ++kb, ++gm) {
                const int s = gm % kStages;
                if (*abort_flag || !mbar_wait(&full[s], (gm / kStages) & 1)) {
                    record_status(status, RFP2_ETIMEOUT);
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a = smem_addr(smem + (size_t)s * kStageBytes);
                const uint64_t adesc = smem_desc_sw128(a);
                const uint64_t bdesc = smem_desc_sw128(a + kABytes);
#pragma unroll
                for (int k = 0; k < BK / UK; ++k)
                    umma_bf16_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc,
                                   (kb > 0 || k > 0) ? 1u : 0u);
                umma_commit_pair_both(&empty[s]);  // both CTAs' stage s free once these complete
            }
            umma_commit_pair_both(&accf[b]);  // accumulator complete (or, after an abort, idle)
        }
    } else if (warp >= 2 && warp < 6) {
        // ---- epilogue (both CTAs): TMEM -> registers -> Y, one tile behind the MMAs.
        // Each 32-row x 32-column chunk goes through a padded shared-memory
        // tile (row = lane on the way in, four rows of 128 bytes per
        // instruction on the way out), so every global store writes whole
        // 128-byte lines instead of 16 bytes in each of 32 rows.
        const int q = warp & 3;  // TMEM lanes 32q .. 32q+31
        float *stg = reinterpret_cast<float *>(smem + Cfg::kStgOff) + (warp - 2) * kStgFloats;
        const uint32_t acce0 = cluster_map(&acce[0], 0);
        int it = 0;
        for (int t = pair; t < nslots; t += npairs, ++it) {
            const int b = it & 1;
            if (*abort_flag || !mbar_wait(&accf[b], (it >> 1) & 1)) {
                record_status(status, RFP2_ETIMEOUT);
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const Slot sl = slot_tile(t, t_full, split_lg, ntm);
            const int row0 = sl.tile_m * PM + (int)rank * BM + q * 32;
            const int nchunks = sl.width / 32;
#pragma unroll 1
            for (int c = 0; c < nchunks; ++c) {
                uint32_t r[32];
                tmem_ld_32cols(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN + c * 32), r);
                tmem_ld_wait();
                float4 *srow = reinterpret_cast<float4 *>(stg + lane * kStgStride);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    srow[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                          __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                __syncwarp();
                const int col = sl.col0 + c * 32 + (lane & 7) * 4;
                float4 cs = make_float4(1.f, 1.f, 1.f, 1.f);
                if (colscale && col < Mw)  // per weight row (e.g. HFP4's row_scale_a)
                    cs = *reinterpret_cast<const float4 *>(colscale + col);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int rr = 4 * j + (lane >> 3);
                    float4 v = *reinterpret_cast<const float4 *>(stg + rr * kStgStride + (lane & 7) * 4);
                    if (colscale) {
                        v.x *= cs.x;
                        v.y *= cs.y;
                        v.z *= cs.z;
                        v.w *= cs.w;
                    }
                    if (row0 + rr < Ntok && col < Mw)
                        *reinterpret_cast<float4 *>(Y + (int64_t)(row0 + rr) * Mw + col) = v;
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acce0 + 8u * b);
        }
    }
    if constexpr (kDecode) {
        if (warp == 6 && lane == 0) {
            // ---- packed-box producer (both CTAs): the rows of this CTA's B half,
            // 256 K per box, in the decoders' order
            pdl_wait();  // W may come from an earlier kernel
            int u = 0;
            bool ok = true;
            for (int t = pair; t < nslots && ok; t += npairs) {
                const Slot sl = slot_tile(t, t_full, split_lg, ntm);
                const int brow = sl.col0 + (int)rank * (sl.width / 2);
                for (int kq = 0; kq < nk / 4; ++kq, ++u) {
                    const int ps = u % kPStages;
                    if (*abort_flag ||
                        (u >= kPStages && !mbar_wait(&pempty[ps], ((u / kPStages) - 1) & 1))) {
                        record_status(status, RFP2_ETIMEOUT);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&pfull[ps], kPBoxBytes);
                    tma_load_2d(pring + (size_t)ps * kPBoxBytes, &wmap, kq * kPBoxRowBytes, brow,
                                &pfull[ps]);
                }
            }
            // boxes still in flight must land before the CTA retires
            for (int i = max(0, u - kPStages); i < u; ++i)
                if (!mbar_wait(&pfull[i % kPStages], (i / kPStages) & 1))
                    record_status(status, RFP2_ETIMEOUT);
        } else if (warp >= 7) {
            // ---- decoders (both CTAs).  Group gi takes K slices gi, gi + 4, ...
            // of every tile (slice gi of each packed box), so the groups' waits
            // and arrivals overlap; thread tig decodes row tig of this CTA's B
            // half: two 10-byte blocks at byte 20 gi of its 80-byte box row,
            // read as two 16-byte words (conflict-free: rows are 80 bytes apart).
            static_assert(kDecodeGroupWarps * 32 == BN / 2, "one B row per decode thread");
            const int gi = (warp - 7) / kDecodeGroupWarps;
            const int row = ((warp - 7) % kDecodeGroupWarps) * 32 + lane;
            const int wq = (20 * gi & 15) >> 2;  // first word of the slice in the 32-byte window
            const uint32_t full0 = cluster_map(&full[0], 0);
            int gbase = 0, ud = 0;  // k-blocks of earlier tiles, boxes decoded
            bool ok = true;
            for (int t = pair; t < nslots && ok; t += npairs, gbase += nk) {
                const bool active = row < slot_tile(t, t_full, split_lg, ntm).width / 2;
                for (int kb = gi; kb < nk; kb += kDecodeGroups, ++ud) {
                    const int gd = gbase + kb, s = gd % kStages, ps = ud % kPStages;
                    bool w_ok = !*abort_flag && mbar_wait(&pfull[ps], (ud / kPStages) & 1);
                    if (gd >= kStages) w_ok = w_ok && mbar_wait(&empty[s], ((gd / kStages) - 1) & 1);
                    if (!__all_sync(0xffffffffu, w_ok)) {
                        if (lane == 0) record_status(status, RFP2_ETIMEOUT);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    if (active) {
                        const uint4 *win = reinterpret_cast<const uint4 *>(
                            pring + (size_t)ps * kPBoxBytes + row * kPBoxRowBytes + ((20 * gi) & ~15));
                        const uint4 q0 = win[0], q1 = win[1];
                        const uint32_t wv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                        uint32_t w[5];
#pragma unroll
                        for (int i = 0; i < 5; ++i)  // wq is warp-uniform: a select, not a local array
                            w[i] = wq == 0 ? wv[i] : wq == 1 ? wv[i + 1] : wq == 2 ? wv[i + 2] : wv[i + 3];
                        // block 0: codes w0, w1, scales in the low half of w2;
                        // block 1: codes bytes 10-17, scales in the high half of w4
                        const uint32_t code[4] = {w[0], w[1], __funnelshift_r(w[2], w[3], 16),
                                                  __funnelshift_r(w[3], w[4], 16)};
                        float sc[4];
                        decode_scale_pair(w[2] & 0xFFFFu, sc[0], sc[1]);
                        decode_scale_pair(w[4] >> 16, sc[2], sc[3]);
                        uint8_t *brow_s = smem + (size_t)s * kStageBytes + kABytes + row * 128;
#pragma unroll
                        for (int h = 0; h < 4; ++h) {  // 16 weights = two 16-byte chunks each
                            uint32_t o[8];
                            decode_half_bf16(code[h], sc[h], o);
                            *reinterpret_cast<uint4 *>(brow_s + (((2 * h) ^ (row & 7)) << 4)) =
                                make_uint4(o[0], o[1], o[2], o[3]);
                            *reinterpret_cast<uint4 *>(brow_s + (((2 * h + 1) ^ (row & 7)) << 4)) =
                                make_uint4(o[4], o[5], o[6], o[7]);
                        }
                    }
                    fence_proxy_async_smem();  // the tensor core reads these bytes next
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive_remote(full0 + 8u * s);
                        mbar_arrive(&pempty[ps]);
                    }
                }
            }
        }
    }
    if (warp == 0 && lane == 0) {
        // The pair commits of the last stages arrive on this CTA's empty
        // barriers (and the other CTA's copies on the even CTA's full
        // barriers): neither CTA may leave before they have.  After an abort,
        // wait for this CTA's own copies instead where it can see them.
        for (int i = max(0, g - kStages); i < g; ++i) {
            const bool done = *abort_flag && rank == 0
                                  ? mbar_wait(&full[i % kStages], (i / kStages) & 1)
                                  : mbar_wait(&empty[i % kStages], (i / kStages) & 1);
            if (!done) record_status(status, RFP2_ETIMEOUT);
        }
    }
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

}  // namespace
}  // namespace rfp2

using namespace rfp2;

// The tiles of the last partial wave run in 2^split_lg parts (1, 2 or 4) when
// that shortens the wave: R tiles in parts of 1/f take ceil(R f / pairs) / f
// tile times.  Returns the whole-tile slots before them (t_full).
static int64_t gemm_split(int64_t ntiles, int pairs, int *split_lg) {
    const int64_t rem = ntiles % pairs;
    *split_lg = 0;
    if (rem == 0) return ntiles;
    double best = 1.0;  // one tile time with no split
    for (int lg = 1; lg <= 2; ++lg) {
        const int64_t f = 1 << lg;
        const double t = (double)((rem * f + pairs - 1) / pairs) / (double)f;
        if (t < best) {
            best = t;
            *split_lg = lg;
        }
    }
    return *split_lg ? ntiles - rem : ntiles;
}

// One GEMM launch: one CTA pair per pair of SMs that can hold one at a time
// (as many as the device reports for this kernel's size), or one per slot
// when there are fewer slots.  kDecode: wmap_h maps the packed ROCmFP2 rows.
template <bool kDecode>
static rfp2_status launch_gemm(const CUtensorMap &xmap, const CUtensorMap &wmap,
                               const CUtensorMap &wmap_h, const CUtensorMap &wmap_q, int64_t N,
                               int64_t M, int64_t K, float *Y, const float *colscale,
                               int32_t *dev_status, cudaStream_t s) {
    using Cfg = GemmCfg<kDecode>;
    static std::mutex mu;
    static int max_pairs[64] = {0};
    const int dev = current_device();
    int pairs = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && max_pairs[dev] > 0) {
            pairs = max_pairs[dev];
        } else {
            if (set_smem_limit(gemm_kernel<kDecode>, (int)Cfg::kSmemBytes) != cudaSuccess)
                return RFP2_ECUDA;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2);
            cfg.blockDim = dim3(Cfg::kThreads);
            cfg.dynamicSmemBytes = Cfg::kSmemBytes;
            if (cudaOccupancyMaxActiveClusters(
                    &pairs, reinterpret_cast<const void *>(gemm_kernel<kDecode>), &cfg) != cudaSuccess ||
                pairs <= 0)
                return RFP2_ECUDA;
            if (dev < 64) max_pairs[dev] = pairs;
        }
    }
    const int64_t tiles = ((N + PM - 1) / PM) * ((M + BN - 1) / BN);
    int split_lg = 0;
    const int64_t t_full = gemm_split(tiles, pairs, &split_lg);
    const int64_t nslots = t_full + ((tiles - t_full) << split_lg);
    const dim3 grid((unsigned)(2 * std::min<int64_t>(nslots, pairs)));
    return from_cuda(launch(gemm_kernel<kDecode>, grid, dim3(Cfg::kThreads), Cfg::kSmemBytes, s, true,
                            xmap, wmap, wmap_h, wmap_q, Y, (int)N, (int)M, (int)K, (int)t_full,
                            split_lg, colscale, dev_status));
}

static bool encode_x_map(CUtensorMap *xmap, const uint16_t *X, int64_t N, int64_t K) {
    return encode_tensor_map_2d(xmap, X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (uint64_t)K, (uint64_t)N,
                                (uint64_t)K * 2, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
}

extern "C" size_t rfp2_gemm_workspace_bytes(int64_t M, int64_t K) {
    (void)M;
    (void)K;
    return 0;
}

extern "C" rfp2_status rfp2_gemm(const uint8_t *W, int64_t M, int64_t K, const uint16_t *X,
                                 int64_t N, float *Y, void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, rfp2_stream_t stream) {
    (void)workspace;
    (void)workspace_bytes;
    if (!W || !X || !Y) return RFP2_EINVAL;
    if (M <= 0 || K <= 0 || N <= 0) return RFP2_ESHAPE;
    if (M > (1LL << 30) || N > (1LL << 30) || K > (1 << 20)) return RFP2_ESHAPE;
    if (K % 256 != 0 || M % 16 != 0) return RFP2_EUNSUPPORTED;
    if (!aligned(W, 16) || !aligned(X, 16) || !aligned(Y, 16)) return RFP2_EALIGN;
    const uint64_t row_bytes = (uint64_t)(K / 32) * 10;  // a multiple of 80
    CUtensorMap xmap, pmap;
    if (!encode_x_map(&xmap, X, N, K) ||
        !encode_tensor_map_2d(&pmap, W, CU_TENSOR_MAP_DATA_TYPE_UINT8, row_bytes, (uint64_t)M,
                              row_bytes, kPBoxRowBytes, BN / 2, CU_TENSOR_MAP_SWIZZLE_NONE))
        return RFP2_ECUDA;
    return launch_gemm<true>(xmap, pmap, pmap, pmap, N, M, K, Y, nullptr, dev_status,
                             reinterpret_cast<cudaStream_t>(stream));
}

// ---- HFP4G32 prefill GEMM ------------------------------------------------------

static size_t hfp4_gemm_ws(int64_t M, int64_t K) {
    return ((size_t)M * K * 2 + 255) / 256 * 256 + (size_t)M * 4;
}

extern "C" size_t hfp4_gemm_workspace_bytes(int64_t M, int64_t K) {
    if (M <= 0 || K <= 0) return 0;
    return hfp4_gemm_ws(M, K);
}

extern "C" rfp2_status hfp4_gemm(const uint8_t *W, int64_t M, int64_t K, const uint16_t *X,
                                 int64_t N, float *Y, void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, rfp2_stream_t stream) {
    if (!W || !X || !Y) return RFP2_EINVAL;
    if (M <= 0 || K <= 0 || N <= 0) return RFP2_ESHAPE;
    if (M > (1LL << 30) || N > (1LL << 30) || K > (1 << 20)) return RFP2_ESHAPE;
    if (K % 256 != 0 || M % 16 != 0) return RFP2_EUNSUPPORTED;
    if (!workspace || workspace_bytes < hfp4_gemm_ws(M, K)) return RFP2_EWORKSPACE;
    if (!aligned(W, 16) || !aligned(X, 16) || !aligned(Y, 16) || !aligned(workspace, 256))
        return RFP2_EALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    __nv_bfloat16 *wexp = static_cast<__nv_bfloat16 *>(workspace);
    float *rs32 = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                            ((size_t)M * K * 2 + 255) / 256 * 256);
    const int KB = (int)(K / 32);
    const int rb = (int)(16 + 17 * KB);
    const int64_t nblocks = M * KB;
    cudaError_t e = launch(hfp4_expand_bf16_kernel, dim3((unsigned)((nblocks + 255) / 256)),
                           dim3(256), 0, s, true, W, (int)M, KB, rb, wexp, rs32);
    if (e != cudaSuccess) return RFP2_ECUDA;
    CUtensorMap xmap, wmap, wmap_h, wmap_q;
    if (!encode_x_map(&xmap, X, N, K) ||
        !encode_tensor_map_2d(&wmap, wexp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (uint64_t)K,
                              (uint64_t)M, (uint64_t)K * 2, BK, BN / 2, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_2d(&wmap_h, wexp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (uint64_t)K,
                              (uint64_t)M, (uint64_t)K * 2, BK, BN / 4, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_2d(&wmap_q, wexp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (uint64_t)K,
                              (uint64_t)M, (uint64_t)K * 2, BK, BN / 8, CU_TENSOR_MAP_SWIZZLE_128B))
        return RFP2_ECUDA;
    return launch_gemm<false>(xmap, wmap, wmap_h, wmap_q, N, M, K, Y, rs32, dev_status, s);
}
