// HFP4G32 GEMV: y[n, m] = row_scale_a(m) * sum_b 2^(e_b - 127) *
// sum_i E2M1[c_i] * x[n, 32b + i], fp32 activations, fp32 accumulation.
//
// Source: "HFP4" (hipfire.dev), sections "Element format (OCP E2M1)",
// "Block scale - UE8M0", "Per-row second-level scale (FP16)" (row_scale_a is
// applied once per row, outside the K loop), "Byte layout - HFP4G32" and
// "Nibble packing"; the page's correctness-anchor loop is the oracle.
//
// GB300 design (the page's kernels are RDNA v_ldexp/WMMA code):
//  * E2M1 codes are exact in f16, so each 32-weight block is two k-steps of
//    m16n8k16 f16 MMAs per row tile with a fresh fp32 accumulator, scaled by
//    2^(e-127) (the block exponent varies per row and block, so it cannot be
//    folded into the accumulation).  The activation columns are the MMA's n
//    dimension, so the weight decode (one E2M1x2 -> f16x2 conversion per two
//    weights) is shared by all columns; for N <= 4 both f16 pieces of every
//    token fit in the eight columns and one MMA per k-step does the block.
//  * fp32 activations are made exact enough for f16 by a prep kernel: each
//    column is scaled by a power of two 2^-kc (max |x| -> [1, 2)) and split
//    into two f16 pieces x' ~= hi + lo (relative residual <= 2^-22); both
//    pieces go through the MMA, and 2^kc is applied with row_scale_a at the
//    end.  The prep kernel writes the pieces in MMA fragment order.
//  * Weights stream through 2-D TMA tiles of 64 rows x 1024 K (544 bytes per
//    row; rows past M and columns past the row are zero-filled), with the
//    matching activation fragments, into a 3-4 stage ring; sixteen consumer
//    warps each take 2 of the 32 blocks of a tile, and their partial sums are
//    combined in shared memory.  All waits are bounded.
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "tma.cuh"

namespace rfp2 {
namespace {

constexpr int kTile = 16;                // MMA rows
constexpr int kMaxTiles = 4;             // row tiles per CTA
constexpr int kRows = kTile * kMaxTiles; // 64 rows per stage
constexpr int kChunkBlocks = 32;         // 1024 K per stage
constexpr int kChunkRowBytes = kChunkBlocks * 17;  // 544
constexpr int kWStageBytes = kRows * kChunkRowBytes;  // 34816
#ifndef RFP2_HFP4_WARPS
#define RFP2_HFP4_WARPS 16
#endif
constexpr int kWarps = RFP2_HFP4_WARPS;  // consumer warps
constexpr int kBlocksPerWarp = kChunkBlocks / kWarps;  // blocks of a chunk per warp
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kRedBytes = kWarps * kMaxTiles * 32 * 16;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// workspace: kc int32 [N] (256 bytes) then fragments uint4 [K/16][N][4]
size_t hfp4_ws_bytes(int64_t N, int64_t K) { return 256 + (size_t)(K / 16) * N * 4 * 16; }

__device__ __forceinline__ uint32_t pack_h2(__half lo, __half hi) {
    return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

// Fragment entry (k-step ks, lane group p) of one column: its four elements
// x * 2^-kc as hi and lo f16 pieces.
__device__ __forceinline__ uint4 split_entry(const float *xr, int kc, int ks, int p) {
    const int base = (ks >> 1) * 32 + 8 * p + 4 * (ks & 1);
    __half h1[4], h2[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float v = ldexpf(xr[base + i], -kc);
        h1[i] = __float2half_rn(v);
        h2[i] = __float2half_rn(v - __half2float(h1[i]));
    }
    return make_uint4(pack_h2(h1[0], h1[1]), pack_h2(h1[2], h1[3]), pack_h2(h2[0], h2[1]),
                      pack_h2(h2[2], h2[3]));
}

// Grid (slices, N): every CTA of column n finds max |x| over the whole column
// (the column is a few KB and read from L2 by each slice), then writes its
// slice of the power-of-two-scaled two-piece f16 split, in the B-fragment
// order of mma.m16n8k16 for the K permutation used by the GEMV (MMA k 2p+i
// <-> element 8p+4s+i and 2p+8+i <-> 8p+4s+2+i of a 32-element block, k-step
// s of the block).
__global__ void __launch_bounds__(256) hfp4_split_kernel(const float *__restrict__ x, int N, int K,
                                                         int *kc_out, uint4 *frag) {
    __shared__ float wmax[8];
    pdl_wait();
    pdl_launch_dependents();
    const int n = blockIdx.y;
    const float *xr = x + (int64_t)n * K;
    float amax = 0.0f;
    if ((reinterpret_cast<uintptr_t>(xr) & 15) == 0) {
        const float4 *x4 = reinterpret_cast<const float4 *>(xr);
        for (int k = threadIdx.x; k < K / 4; k += blockDim.x) {
            const float4 v = __ldg(x4 + k);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
    } else {
        for (int k = threadIdx.x; k < K; k += blockDim.x) amax = fmaxf(amax, fabsf(__ldg(xr + k)));
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, wmax[i]);
    const int kc = amax > 0.0f ? ilogbf(amax) : 0;  // max |x| * 2^-kc in [1, 2)
    if (threadIdx.x == 0 && blockIdx.x == 0) kc_out[n] = kc;
    const int entries = (K / 16) * 4;
    const int per = (entries + gridDim.x - 1) / gridDim.x;
    const int e0 = blockIdx.x * per, e1 = min(entries, e0 + per);
    for (int e = e0 + threadIdx.x; e < e1; e += blockDim.x)
        frag[((int64_t)(e >> 2) * N + n) * 4 + (e & 3)] = split_entry(xr, kc, e >> 2, e & 3);
}

// Eight E2M1 codes (four bytes; in each byte the low nibble is the even
// element) -> four f16x2 words (low half = even element).
__device__ __forceinline__ void e2m1x8_to_h2x4(uint32_t w, uint32_t &h0, uint32_t &h1,
                                               uint32_t &h2, uint32_t &h3) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// UE8M0 byte -> 2^(e-127) as fp32 (e = 0 is the subnormal 2^-127, 0xFF NaN).
__device__ __forceinline__ float ue8m0(uint32_t e) {
    uint32_t bits = e << 23;
    bits = e == 0 ? 0x00400000u : bits;
    bits = e == 0xFF ? 0x7FC00000u : bits;
    return __uint_as_float(bits);
}

// Four bytes of a row starting at an arbitrary byte address in shared memory.
__device__ __forceinline__ uint32_t load_u32_unaligned(const uint8_t *p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t *w = reinterpret_cast<const uint32_t *>(a & ~uintptr_t(3));
    return __funnelshift_r(w[0], w[1], (uint32_t)(a & 3) * 8);
}

struct HfpArgs {
    const uint8_t *W;
    int M, K, N, rb;
    int tiles_per_cta, tiles_extra, nstages;
    float *y;
    int32_t *status;
    const int *kc;
    const uint4 *frag;
    const float *x;  // FOLD: the activations themselves
    int w_early;     // FOLD: stream W before the earlier work has completed
};

// PAIRED (N <= 4): the two f16 pieces of token n are MMA columns 2n and
// 2n + 1, so one MMA per k-step covers both; otherwise the columns are the
// tokens and each piece takes its own MMA.  FOLD (small N * K): the consumer
// warps build the fragments of the whole K in shared memory themselves (the
// split kernel's arithmetic), so no split launch precedes the GEMV.
template <bool PAIRED, bool FOLD>
__global__ void __launch_bounds__(kThreads, 1)
    hfp4_gemv_kernel(const __grid_constant__ CUtensorMap wmap, HfpArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int S = a.nstages;
    const int bstage_bytes = 64 * a.N * 64;  // 64 k-steps x N columns x 4 lanes x 16 B
    uint8_t *wst = smem;                                        // [S][kWStageBytes]
    uint8_t *bst = smem + (size_t)S * kWStageBytes;             // [S][bstage_bytes], FOLD: [K/16][N][4]
    const size_t bbytes = FOLD ? (size_t)(a.K / 16) * a.N * 64 : (size_t)S * bstage_bytes;
    float *red = reinterpret_cast<float *>(bst + bbytes);  // [8][4][32][4]
    __shared__ int kc_s[RFP2_MAX_BATCH];
    __shared__ float cmax[kWarps];
    uint64_t *full = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(red) + kRedBytes);
    uint64_t *empty = full + S;
    uint64_t *red_bar = empty + S;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(red_bar + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bx = blockIdx.x;
    const int tile0 = bx * a.tiles_per_cta + min(bx, a.tiles_extra);
    const int ntiles = a.tiles_per_cta + (bx < a.tiles_extra ? 1 : 0);
    const int row0 = tile0 * kTile;
    const int KB = a.K >> 5;
    const int nchunks = (KB + kChunkBlocks - 1) / kChunkBlocks;
    const int nks = a.K / 16;

    // 2^(e-127) for every UE8M0 byte (0 -> 2^-127, 0xFF -> NaN)
    __shared__ float scale_lut[256];
    for (int e = threadIdx.x; e < 256; e += blockDim.x) scale_lut[e] = ue8m0((uint32_t)e);
    if (threadIdx.x == kWarps * 32) {
        prefetch_tensor_map(&wmap);
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        mbar_init(red_bar, kWarps);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kWarps) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int c = 0;
            // Without FOLD the split kernel of this call ran first and only
            // released this launch after the earlier work had completed, so
            // the weight tiles can start at once.  With FOLD this is the
            // call's only kernel: W is read before that point only when the
            // caller turned weight prefetch on.
            if (FOLD && !a.w_early) pdl_wait();
            for (; c < nchunks && c < S; ++c) {
                const int ks0 = c * 2 * kChunkBlocks;
                const int bbytes = FOLD ? 0 : min(2 * kChunkBlocks, nks - ks0) * a.N * 64;
                mbar_arrive_expect_tx(&full[c], kWStageBytes + bbytes);
                tma_load_2d_hint(wst + (size_t)c * kWStageBytes, &wmap, 4 + c * (kChunkRowBytes / 4),
                                 row0, &full[c], pol);
            }
            if (!FOLD) {
                pdl_wait();  // the activation fragments come from the split kernel
                for (int i = 0; i < c; ++i) {
                    const int ks0 = i * 2 * kChunkBlocks;
                    const int bbytes = min(2 * kChunkBlocks, nks - ks0) * a.N * 64;
                    bulk_g2s(bst + (size_t)i * bstage_bytes, a.frag + (int64_t)ks0 * a.N * 4, bbytes,
                             &full[i]);
                }
            }
            for (; c < nchunks; ++c) {
                const int s = c % S;
                if (!mbar_wait(&empty[s], ((c / S) - 1) & 1)) {
                    record_status(a.status, RFP2_ETIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                const int ks0 = c * 2 * kChunkBlocks;
                const int bbytes = FOLD ? 0 : min(2 * kChunkBlocks, nks - ks0) * a.N * 64;
                mbar_arrive_expect_tx(&full[s], kWStageBytes + bbytes);
                tma_load_2d_hint(wst + (size_t)s * kWStageBytes, &wmap, 4 + c * (kChunkRowBytes / 4),
                                 row0, &full[s], pol);
                if (!FOLD)
                    bulk_g2s(bst + (size_t)s * bstage_bytes, a.frag + (int64_t)ks0 * a.N * 4, bbytes,
                             &full[s]);
            }
            // no copy may be in flight when the CTA exits: without an abort
            // every consumer warp waits for every chunk before it finishes,
            // so only an aborted CTA waits here for its last copies
            if (*abort_flag == 0) return;
            for (int i = max(0, c - S); i < c; ++i)
                if (!mbar_wait(&full[i % S], (i / S) & 1)) record_status(a.status, RFP2_ETIMEOUT);
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    pdl_wait();
    pdl_launch_dependents();
    if constexpr (FOLD) {
        // per column: kc from max |x| (scaled values below 2), then every
        // fragment entry of the whole K
        const int ct = threadIdx.x;  // 0 .. kWarps*32-1
        for (int n = 0; n < a.N; ++n) {
            const float *xr = a.x + (int64_t)n * a.K;
            float amax = 0.0f;
            for (int k = ct; k < a.K; k += kWarps * 32) amax = fmaxf(amax, fabsf(xr[k]));
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            if (lane == 0) cmax[warp] = amax;
            named_bar_sync(1, kWarps * 32);
            if (ct == 0) {
                float m = 0.0f;
                for (int w = 0; w < kWarps; ++w) m = fmaxf(m, cmax[w]);
                kc_s[n] = m > 0.0f ? ilogbf(m) : 0;
            }
            named_bar_sync(1, kWarps * 32);
        }
        uint4 *fr = reinterpret_cast<uint4 *>(bst);
        const int entries = nks * 4 * a.N;
        for (int e = ct; e < entries; e += kWarps * 32) {
            const int p = e & 3, n = (e >> 2) % a.N, ks = (e >> 2) / a.N;
            fr[e] = split_entry(a.x + (int64_t)n * a.K, kc_s[n], ks, p);
        }
        named_bar_sync(1, kWarps * 32);
    }
    const int g = lane >> 2, p = lane & 3;
    float acc[kMaxTiles][4];
#pragma unroll
    for (int t = 0; t < kMaxTiles; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][i] = 0.0f;
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
        const int s = c % S;
        if (*abort_flag || !mbar_wait(&full[s], (c / S) & 1)) {
            record_status(a.status, RFP2_ETIMEOUT);
            *abort_flag = 1;
            ok = false;
            break;
        }
        const uint8_t *ws = wst + (size_t)s * kWStageBytes;
        const uint4 *bs = FOLD ? reinterpret_cast<const uint4 *>(bst) + (size_t)c * 2 * kChunkBlocks * a.N * 4
                               : reinterpret_cast<const uint4 *>(bst + (size_t)s * bstage_bytes);
#pragma unroll
        for (int jj = 0; jj < kBlocksPerWarp; ++jj) {
            const int j = warp * kBlocksPerWarp + jj;  // block inside the chunk
            if (c * kChunkBlocks + j >= KB) break;
            uint32_t b[4] = {0u, 0u, 0u, 0u};  // k-step 0 (b[0], b[1]), k-step 1 (b[2], b[3])
            if constexpr (PAIRED) {
                const int n = g >> 1;
                if (n < a.N) {
                    const uint4 t0 = bs[((2 * j) * a.N + n) * 4 + p];
                    const uint4 t1 = bs[((2 * j + 1) * a.N + n) * 4 + p];
                    const bool lo = (g & 1) != 0;
                    b[0] = lo ? t0.z : t0.x;
                    b[1] = lo ? t0.w : t0.y;
                    b[2] = lo ? t1.z : t1.x;
                    b[3] = lo ? t1.w : t1.y;
                }
            }
            uint4 b0 = make_uint4(0, 0, 0, 0), b1 = make_uint4(0, 0, 0, 0);
            if constexpr (!PAIRED) {
                if (g < a.N) {
                    b0 = bs[((2 * j) * a.N + g) * 4 + p];
                    b1 = bs[((2 * j + 1) * a.N + g) * 4 + p];
                }
            }
#pragma unroll
            for (int t = 0; t < kMaxTiles; ++t) {
                if (t < ntiles) {
                    const uint8_t *ra = ws + (t * kTile + g) * kChunkRowBytes + j * 17;
                    const uint8_t *rbp = ra + 8 * kChunkRowBytes;
                    const uint32_t wa = load_u32_unaligned(ra + 1 + 4 * p);
                    const uint32_t wb = load_u32_unaligned(rbp + 1 + 4 * p);
                    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    // k-step 0: bytes 0,1 of the word; k-step 1: bytes 2,3
                    uint32_t a0, a1, a2, a3, a4, a5, a6, a7;
                    e2m1x8_to_h2x4(wa, a0, a2, a4, a6);
                    e2m1x8_to_h2x4(wb, a1, a3, a5, a7);
                    const float sa = scale_lut[ra[0]], sb = scale_lut[rbp[0]];
                    if constexpr (PAIRED) {
                        mma_f16(d, a0, a1, a2, a3, b[0], b[1]);
                        mma_f16(d, a4, a5, a6, a7, b[2], b[3]);
                        // columns 2p, 2p+1 = the two pieces of token p
                        acc[t][0] = fmaf(d[0] + d[1], sa, acc[t][0]);
                        acc[t][1] = fmaf(d[2] + d[3], sb, acc[t][1]);
                    } else {
                        mma_f16(d, a0, a1, a2, a3, b0.x, b0.y);
                        mma_f16(d, a0, a1, a2, a3, b0.z, b0.w);
                        mma_f16(d, a4, a5, a6, a7, b1.x, b1.y);
                        mma_f16(d, a4, a5, a6, a7, b1.z, b1.w);
                        acc[t][0] = fmaf(d[0], sa, acc[t][0]);
                        acc[t][1] = fmaf(d[1], sa, acc[t][1]);
                        acc[t][2] = fmaf(d[2], sb, acc[t][2]);
                        acc[t][3] = fmaf(d[3], sb, acc[t][3]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    // combine the eight K-slices: every warp writes its partials, warp 0 sums
    float4 *red4 = reinterpret_cast<float4 *>(red);
#pragma unroll
    for (int t = 0; t < kMaxTiles; ++t)
        red4[(warp * kMaxTiles + t) * 32 + lane] = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
    __syncwarp();
    if (lane == 0) mbar_arrive(red_bar);
    if (warp != 0) return;
    if (!mbar_wait(red_bar, 0)) {
        record_status(a.status, RFP2_ETIMEOUT);
        return;
    }
    if (!ok) return;
    for (int t = 0; t < ntiles; ++t) {
        float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int w = 0; w < kWarps; ++w) {
            const float4 q = red4[(w * kMaxTiles + t) * 32 + lane];
            v[0] += q.x;
            v[1] += q.y;
            v[2] += q.z;
            v[3] += q.w;
        }
        const int r0 = row0 + t * kTile + g, r1 = r0 + 8;
        const float rs0 =
            r0 < a.M ? __half2float(*reinterpret_cast<const __half *>(a.W + (int64_t)r0 * a.rb)) : 0.0f;
        const float rs1 =
            r1 < a.M ? __half2float(*reinterpret_cast<const __half *>(a.W + (int64_t)r1 * a.rb)) : 0.0f;
        if constexpr (PAIRED) {
            if (p < a.N) {
                const float s0 = ldexpf(1.0f, FOLD ? kc_s[p] : a.kc[p]);
                if (r0 < a.M) a.y[(int64_t)p * a.M + r0] = v[0] * rs0 * s0;
                if (r1 < a.M) a.y[(int64_t)p * a.M + r1] = v[1] * rs1 * s0;
            }
        } else {
            const int c0 = 2 * p, c1 = 2 * p + 1;
            const float s0 = c0 < a.N ? ldexpf(1.0f, FOLD ? kc_s[c0] : a.kc[c0]) : 0.0f;
            const float s1 = c1 < a.N ? ldexpf(1.0f, FOLD ? kc_s[c1] : a.kc[c1]) : 0.0f;
            if (r0 < a.M) {
                if (c0 < a.N) a.y[(int64_t)c0 * a.M + r0] = v[0] * rs0 * s0;
                if (c1 < a.N) a.y[(int64_t)c1 * a.M + r0] = v[1] * rs0 * s1;
            }
            if (r1 < a.M) {
                if (c0 < a.N) a.y[(int64_t)c0 * a.M + r1] = v[2] * rs1 * s0;
                if (c1 < a.N) a.y[(int64_t)c1 * a.M + r1] = v[3] * rs1 * s1;
            }
        }
    }
}

}  // namespace
}  // namespace rfp2

using namespace rfp2;

extern "C" size_t hfp4_gemv_workspace_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0) return 0;
    return hfp4_ws_bytes(N, K);
}

extern "C" rfp2_status hfp4_gemv(const uint8_t *W, int64_t M, int64_t K, const float *x, int64_t N,
                                 float *y, void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, rfp2_stream_t stream) {
    if (!W || !x || !y) return RFP2_EINVAL;
    if (M <= 0 || K <= 0 || N < 1 || N > RFP2_MAX_BATCH) return RFP2_ESHAPE;
    if (M > (1 << 30) || K > (1 << 24)) return RFP2_ESHAPE;
    if (K % 512 != 0) return RFP2_EUNSUPPORTED;  // rows must be whole 16-byte units
    if (!workspace || workspace_bytes < hfp4_ws_bytes(N, K)) return RFP2_EWORKSPACE;
    if (!aligned(W, 16) || !aligned(x, 4) || !aligned(y, 4) || !aligned(workspace, 256))
        return RFP2_EALIGN;
    const int rb = (int)(16 + 17 * (K / 32));
    CUtensorMap wmap;
    if (!encode_tensor_map_2d(&wmap, W, CU_TENSOR_MAP_DATA_TYPE_UINT32, (uint64_t)rb / 4,
                              (uint64_t)M, (uint64_t)rb, kChunkRowBytes / 4, kRows))
        return RFP2_ECUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int *kc = static_cast<int *>(workspace);
    uint4 *frag = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(workspace) + 256);
    // Small N * K: the GEMV builds the fragments itself (no split launch, no
    // dependency hop); they stay in shared memory for the whole K.
    const size_t fold_bytes = (size_t)(K / 16) * N * 64;
    const bool fold = N <= 2 && fold_bytes <= 64 * 1024;
    if (!fold) {
        // slices of K per column: about 1024 fragment entries (4096 elements) each
        const int slices = (int)std::min<int64_t>(64, std::max<int64_t>(1, K / 4096));
        cudaError_t e = launch(hfp4_split_kernel, dim3((unsigned)slices, (unsigned)N), dim3(256), 0,
                               s, true, x, (int)N, (int)K, kc, frag);
        if (e != cudaSuccess) return RFP2_ECUDA;
    }
    // stages: as many 64-row x 1024-K tiles (plus their fragments) as fit
    const size_t per_stage = kWStageBytes + (fold ? 0 : (size_t)64 * N * 64);
    const size_t fixed = (fold ? fold_bytes : 0) + kRedBytes + 256;
    int stages = 4;
    while (stages > 2 && stages * per_stage + fixed > 224 * 1024) --stages;
    const size_t smem = stages * per_stage + fixed;
    static std::mutex mu;
    static int configured[64] = {0};
    const int dev = current_device();
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && !configured[dev]) {
            if (set_smem_limit(hfp4_gemv_kernel<true, false>, 224 * 1024) != cudaSuccess ||
                set_smem_limit(hfp4_gemv_kernel<false, false>, 224 * 1024) != cudaSuccess ||
                set_smem_limit(hfp4_gemv_kernel<true, true>, 224 * 1024) != cudaSuccess)
                return RFP2_ECUDA;
            configured[dev] = 1;
        }
    }
    const int tiles = (int)((M + kTile - 1) / kTile);
    int grid = sm_count(dev);
    if (grid > tiles) grid = tiles;
    while ((tiles + grid - 1) / grid > kMaxTiles) ++grid;
    HfpArgs a;
    a.W = W;
    a.M = (int)M;
    a.K = (int)K;
    a.N = (int)N;
    a.rb = rb;
    a.tiles_per_cta = tiles / grid;
    a.tiles_extra = tiles % grid;
    a.nstages = stages;
    a.y = y;
    a.status = dev_status;
    a.kc = kc;
    a.frag = frag;
    a.x = x;
    a.w_early = weight_prefetch() ? 1 : 0;
    if (fold)
        return from_cuda(launch(hfp4_gemv_kernel<true, true>, dim3(grid), dim3(kThreads), smem, s,
                                true, wmap, a));
    if (N <= 4)
        return from_cuda(launch(hfp4_gemv_kernel<true, false>, dim3(grid), dim3(kThreads), smem, s,
                                true, wmap, a));
    return from_cuda(launch(hfp4_gemv_kernel<false, false>, dim3(grid), dim3(kThreads), smem, s,
                            true, wmap, a));
}
