// Block-scaled FP4 (NVFP4) form of the ROCmFP2 prefill GEMM: ROCmFP2 weights
// are exactly NVFP4 blocks, so with NVFP4 activations the product runs on the
// FP4 tensor cores (tcgen05.mma kind::mxf4nvf4, 16-element blocks, E4M3
// scales).
//
// Source: "ROCmFP2 codebook research report", section "02 Quantization": the
// UE4M3 scale s(b) is half the E4M3FN value of the same byte, so a weight
// codebook[c] * s(b) = (codebook[c] / 2) * E4M3FN(b), and codebook / 2 is in
// {-2, -0.5, +0.5, +2}: E2M1 values.  The "HFP4" page names NVIDIA NVFP4 (G16
// / E4M3 scaling) as the reference format; the activation recipe below is
// NVIDIA's published one (a per-token fp32 factor g = 448 * 6 / amax, a
// per-16 E4M3 scale of (bmax / 6) * g, E2M1 elements), so this path is not
// exact on the activation side: it has its own tolerance.
//
// GB300 design.
//  * Weights convert once (like packing) into an NVFP4 image: E2M1 codes [M,
//    K/2] (element 2j in the low nibble of byte j) followed by the scale
//    bytes [M, K/16], which are the ROCmFP2 scale bytes unchanged.
//  * Activations (bf16 tokens) are quantized per call into the workspace:
//    codes [N, K/2], scale bytes [N, K/16], g [N].
//  * The GEMM is persistent over 128-weight-row x 128-token tiles.  A TMA
//    warp streams 128-byte-wide (256-element) K stages of both code matrices
//    with the 128-byte swizzle the MMA descriptors expect, and the stage's
//    16 scale bytes of every row and token beside them; four scale warps
//    copy each stage's scale bytes into tensor memory in the layout the
//    block-scaled MMA reads (for one MMA of K = 64 the four bytes of row or
//    token (L % 32) + 32q sit in lane L, every lane quadrant, column base +
//    q); one thread issues four kind::mxf4nvf4 MMAs per stage into one of two
//    128-column fp32 accumulators; four epilogue warps read the finished
//    accumulator, multiply by the token's 1/g and store y (consecutive
//    weight rows in consecutive lanes: coalesced).
//  * Every wait is bounded; a timeout records RFP2_ETIMEOUT and the CTA
//    winds down after its tensor-core work and copies have completed.
#include <cuda_fp16.h>

#include <mutex>

#include "common.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace rfp2 {
namespace {

// ---------------------------------------------------------------------------
// Weight conversion.  Byte c of the table is the E2M1 code of codebook[c] / 2:
// code 0 (-4) -> -2 (0xC), 1 (-1) -> -0.5 (0x9), 2 (+1) -> +0.5 (0x1),
// 3 (+4) -> +2 (0x4).
constexpr uint32_t kNvTable = 0x0401090Cu;

// Sixteen 2-bit codes (code i at bits 2i, 2i+1) -> sixteen E2M1 nibbles
// (element 2j in the low nibble of byte j): lo = codes 0..7, hi = 8..15.
RFP2_DEV void nv_expand16(uint32_t c, uint32_t &lo, uint32_t &hi) {
    const uint32_t s = c & 0x33333333u;          // nibble k: code 2k
    const uint32_t t = (c >> 2) & 0x33333333u;   // nibble k: code 2k + 1
    uint32_t e, o;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(e) : "r"(kNvTable), "r"(s));
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(o) : "r"(kNvTable), "r"(t));
    lo = e | (o << 4);
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(e) : "r"(kNvTable), "r"(s >> 16));
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(o) : "r"(kNvTable), "r"(t >> 16));
    hi = e | (o << 4);
}

// One thread per 10-byte block.
__global__ void nv_convert_kernel(const uint8_t *__restrict__ W, int64_t nblocks, int64_t KB,
                                  uint8_t *__restrict__ codes, uint8_t *__restrict__ sbytes) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nblocks) return;
    const uint16_t *b = reinterpret_cast<const uint16_t *>(W + i * 10);  // 2-byte aligned
    const uint32_t c0 = (uint32_t)b[0] | ((uint32_t)b[1] << 16);
    const uint32_t c1 = (uint32_t)b[2] | ((uint32_t)b[3] << 16);
    uint4 o;
    nv_expand16(c0, o.x, o.y);
    nv_expand16(c1, o.z, o.w);
    // block i of row m = i / KB sits at codes[m, 32 kb / 2] = codes + 16 i
    *reinterpret_cast<uint4 *>(codes + i * 16) = o;
    *reinterpret_cast<uint16_t *>(sbytes + i * 2) = b[4];
    (void)KB;
}

// ---------------------------------------------------------------------------
// Activation quantizer, one CTA of kQThreads per token row.  Per row: amax,
// g = 2688 / amax (1 for an all-zero row); per 16 values t = (bmax / 6) * g,
// scale byte = E4M3 of t rounded to nearest even and saturating at 448
// (cvt.rn.satfinite), s = its value; element code = E2M1 of (x * g) / s,
// nearest even, saturating at 6, with the sign bit of the quotient; a block
// whose scale byte is 0 stores +0.  Every step is an IEEE fp32 operation in
// the order written (no contraction).
constexpr int kQThreads = 256;

RFP2_DEV uint32_t e4m3_rn_sat(float t) {
    uint32_t r;
    asm("{\n .reg .b16 h;\n cvt.rn.satfinite.e4m3x2.f32 h, %1, %2;\n cvt.u32.u16 %0, h;\n}\n"
        : "=r"(r)
        : "f"(0.0f), "f"(t));
    return r & 0xFFu;  // t in the low byte
}
RFP2_DEV float e4m3_value(uint32_t b) {
    uint32_t h2;
    asm("{\n .reg .b16 h;\n cvt.u16.u32 h, %1;\n cvt.rn.f16x2.e4m3x2 %0, h;\n}\n" : "=r"(h2) : "r"(b));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}
// E2M1 magnitude code of |v| (nearest even, saturating at 6), 0..7.
RFP2_DEV uint32_t e2m1_mag(float v) {
    uint32_t r;
    asm("{\n .reg .b8 q;\n cvt.rn.satfinite.e2m1x2.f32 q, %1, %2;\n cvt.u32.u8 %0, q;\n}\n"
        : "=r"(r)
        : "f"(0.0f), "f"(fabsf(v)));
    return r & 0x7u;
}

// bf16 bits of 16 consecutive values -> fp32.
RFP2_DEV void load_block16(const uint16_t *p, float (&f)[16]) {
    const uint4 v0 = *reinterpret_cast<const uint4 *>(p);
    const uint4 v1 = *reinterpret_cast<const uint4 *>(p + 8);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// One 16-value block with the row factor g: scale byte and 16 codes.
RFP2_DEV void quant_block16(const float (&f)[16], float g, uint8_t *codes, uint8_t *sbyte) {
    float bmax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(f[i]));
    const float t = __fmul_rn(__fdiv_rn(bmax, 6.0f), g);
    const uint32_t b = e4m3_rn_sat(t);
    const float s = e4m3_value(b);
    uint32_t out[2] = {0u, 0u};
    if (s != 0.0f) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float e = __fdiv_rn(__fmul_rn(f[i], g), s);
            const uint32_t c = e2m1_mag(e) | (signbit(e) ? 8u : 0u);
            out[i / 8] |= c << (4 * (i % 8));
        }
    }
    *reinterpret_cast<uint2 *>(codes) = make_uint2(out[0], out[1]);
    *sbyte = (uint8_t)b;
}

// The first kQCache blocks of a thread stay in registers between the amax
// pass and the quantization (a row of K <= 16 * kQThreads * kQCache values is
// read once); blocks beyond them are read again.
constexpr int kQCache = 2;

__global__ void __launch_bounds__(kQThreads) nv_quant_kernel(const uint16_t *__restrict__ X, int K,
                                                             uint8_t *__restrict__ codes,
                                                             uint8_t *__restrict__ sbytes,
                                                             float *__restrict__ g_out) {
    __shared__ float red[kQThreads / 32];
    pdl_launch_dependents();
    pdl_wait();
    const int64_t n = blockIdx.x;
    const uint16_t *x = X + n * K;
    const int nb = K / 16;
    float f[kQCache][16];
    float m = 0.0f;
#pragma unroll
    for (int c = 0; c < kQCache; ++c) {
        const int j = threadIdx.x + c * kQThreads;
        if (j < nb) {
            load_block16(x + j * 16, f[c]);
#pragma unroll
            for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(f[c][i]));
        }
    }
    for (int j = threadIdx.x + kQCache * kQThreads; j < nb; j += kQThreads) {
        float t[16];
        load_block16(x + j * 16, t);
#pragma unroll
        for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(t[i]));
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    float amax = red[0];
#pragma unroll
    for (int i = 1; i < kQThreads / 32; ++i) amax = fmaxf(amax, red[i]);
    const float g = amax > 0.0f ? __fdiv_rn(2688.0f, amax) : 1.0f;
    if (threadIdx.x == 0) g_out[n] = g;
#pragma unroll
    for (int c = 0; c < kQCache; ++c) {
        const int j = threadIdx.x + c * kQThreads;
        if (j < nb) quant_block16(f[c], g, codes + n * (K / 2) + j * 8, sbytes + n * (K / 16) + j);
    }
    for (int j = threadIdx.x + kQCache * kQThreads; j < nb; j += kQThreads) {
        float t[16];
        load_block16(x + j * 16, t);
        quant_block16(t, g, codes + n * (K / 2) + j * 8, sbytes + n * (K / 16) + j);
    }
}

// ---------------------------------------------------------------------------
// GEMM.  Tile: 128 weight rows (MMA M) x 128 tokens (MMA N); a stage is 128
// bytes of K (256 elements) of both operands, four MMAs of K = 64.
constexpr int kBM = 128, kBN = 128;
constexpr int kBKB = 128;  // bytes of K per stage
constexpr int kSteps = 4;  // MMAs per stage
constexpr int kNvStages = 6;
constexpr uint32_t kTileBytes = kBM * kBKB;  // 16 KB, the same for the token tile
constexpr uint32_t kSfTileBytes = kBM * 16;  // 16 scale bytes of each of 128 rows
// stage: weight codes, token codes, weight scales, token scales
constexpr uint32_t kStageBytes = 2 * kTileBytes + 2 * kSfTileBytes;
constexpr uint32_t kNvTmemCols = 512;
constexpr uint32_t kAccCols = kBN;              // fp32 columns of one accumulator
constexpr uint32_t kSfCol0 = 2 * kAccCols;      // scale slots after the two accumulators
constexpr uint32_t kSfColsPerStage = 32;        // 16 for the weights, 16 for the tokens
constexpr int kNvThreads = 320;                 // TMA, MMA, 4 scale, 4 epilogue warps
constexpr size_t kNvBarBytes = 256;
constexpr size_t kNvSmem = kNvStages * kStageBytes + kNvBarBytes + 1024;
static_assert(kSfCol0 + kNvStages * kSfColsPerStage <= kNvTmemCols, "tensor memory");
static_assert((3 * kNvStages + 4) * 8 + 8 <= kNvBarBytes, "barrier area");
// kind::mxf4nvf4 instruction descriptor: A and B E2M1 (format 1, bits 7-9 and
// 10-12), both K-major, N >> 3 in bits 17-22, UE4M3 scales (bit 23 = 0),
// M >> 4 in bits 24-28, scale-factor ids 0.
constexpr uint32_t kNvIdesc =
    (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);

// D[tmem] (+)= A * B^T with per-16 E4M3 scales of A rows and B columns read
// from tensor memory at sfa / sfb (issued by one thread).
RFP2_DEV void umma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                        uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
        "[%4], [%5], p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane.
RFP2_DEV void tmem_st_16cols(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// The 16 scale words a lane writes for one stage, from the stage's scale
// tile in shared memory (row r of the tile: its 16 bytes): column 4h + q
// holds the four bytes of K-step h of row lane + 32q, bytes 4h .. 4h+3 of
// that row.  The 32 lanes read 512 consecutive bytes per q.
RFP2_DEV void stage_scales(const uint8_t *tile, int lane, uint32_t (&v)[16]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 u = *reinterpret_cast<const uint4 *>(tile + (lane + 32 * q) * 16);
        v[q] = u.x;
        v[4 + q] = u.y;
        v[8 + q] = u.z;
        v[12 + q] = u.w;
    }
}

__global__ void __launch_bounds__(kNvThreads, 1)
    nv_gemm_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                   const __grid_constant__ CUtensorMap wsmap, const __grid_constant__ CUtensorMap xsmap,
                   const float *__restrict__ g, float *__restrict__ Y, int M, int N, int K,
                   int32_t *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kNvStages * kStageBytes);
    uint64_t *empty = full + kNvStages;
    uint64_t *sf_full = empty + kNvStages;
    uint64_t *acc_full = sf_full + kNvStages;  // [2]
    uint64_t *acc_empty = acc_full + 2;        // [2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntm = (M + kBM - 1) / kBM, ntn = (N + kBN - 1) / kBN;
    const int ntiles = ntm * ntn, nk = K / (2 * kBKB);

    if (threadIdx.x == 0) {
        prefetch_tensor_map(&wmap);
        prefetch_tensor_map(&xmap);
        prefetch_tensor_map(&wsmap);
        prefetch_tensor_map(&xsmap);
        for (int s = 0; s < kNvStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sf_full[s], 4);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kNvTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();
    pdl_wait();  // the token codes, scales and g come from the kernel before

    auto fail = [&]() {
        record_status(status, RFP2_ETIMEOUT);
        *abort_flag = 1;
    };

    if (warp == 0) {
        // ---- TMA producer (one thread)
        if (lane == 0) {
            int gs = 0;
            for (int t = blockIdx.x; t < ntiles && !*abort_flag; t += gridDim.x) {
                const int tm = t % ntm, tn = t / ntm;
                for (int kk = 0; kk < nk; ++kk, ++gs) {
                    const int s = gs % kNvStages;
                    if (gs >= kNvStages && !mbar_wait(&empty[s], ((gs / kNvStages) - 1) & 1)) {
                        fail();
                        break;
                    }
                    if (*abort_flag) break;
                    mbar_arrive_expect_tx(&full[s], kStageBytes);
                    uint8_t *st = smem + (size_t)s * kStageBytes;
                    tma_load_2d(st, &wmap, kk * kBKB, tm * kBM, &full[s]);
                    tma_load_2d(st + kTileBytes, &xmap, kk * kBKB, tn * kBN, &full[s]);
                    tma_load_2d(st + 2 * kTileBytes, &wsmap, kk * 16, tm * kBM, &full[s]);
                    tma_load_2d(st + 2 * kTileBytes + kSfTileBytes, &xsmap, kk * 16, tn * kBN, &full[s]);
                }
            }
            // every copy in flight lands before the CTA may exit
            for (int i = gs > kNvStages ? gs - kNvStages : 0; i < gs; ++i)
                if (!mbar_wait(&full[i % kNvStages], (i / kNvStages) & 1)) fail();
        }
    } else if (warp == 1) {
        // ---- MMA issuer (the whole warp; one elected lane issues)
        int gs = 0, it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++it) {
            const int b = it & 1;
            if (it >= 2 && (*abort_flag || !mbar_wait(&acc_empty[b], ((it >> 1) - 1) & 1))) {
                fail();
                ok = false;
                break;
            }
            for (int kk = 0; kk < nk; ++kk, ++gs) {
                const int s = gs % kNvStages;
                const uint32_t ph = (gs / kNvStages) & 1;
                if (*abort_flag || !mbar_wait(&full[s], ph) || !mbar_wait(&sf_full[s], ph)) {
                    fail();
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    const uint32_t sa = smem_addr(smem + (size_t)s * kStageBytes);
                    const uint64_t ad = smem_desc_sw128(sa), bd = smem_desc_sw128(sa + kTileBytes);
                    const uint32_t sfa = tmem + kSfCol0 + s * kSfColsPerStage;
#pragma unroll
                    for (int h = 0; h < kSteps; ++h)
                        umma_nvf4(tmem + b * kAccCols, ad + 2 * h, bd + 2 * h, kNvIdesc, sfa + 4 * h,
                                  sfa + 16 + 4 * h, (kk | h) != 0 ? 1u : 0u);
                    umma_commit(&empty[s]);
                }
                __syncwarp();
            }
            if (!ok) break;
            if (elect_one()) umma_commit(&acc_full[b]);
            __syncwarp();
        }
        // the tensor cores finish every issued MMA before the memory is freed
        if (gs > 0 && !mbar_wait(&empty[(gs - 1) % kNvStages], ((gs - 1) / kNvStages) & 1)) fail();
    } else if (warp < 6) {
        // ---- scale warps: this warp's lane quadrant of every scale slot.  A
        // stage's copies land only after the MMAs of the slot's previous
        // round have completed (the producer waited for that), so the slot's
        // tensor memory is free once the stage is full.
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        int gs = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            for (int kk = 0; kk < nk; ++kk, ++gs) {
                const int s = gs % kNvStages;
                if (*abort_flag || !mbar_wait(&full[s], (gs / kNvStages) & 1)) {
                    fail();
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t *st = smem + (size_t)s * kStageBytes + 2 * kTileBytes;
                uint32_t va[16], vb[16];
                stage_scales(st, lane, va);
                stage_scales(st + kSfTileBytes, lane, vb);
                const uint32_t col = tmem + lane_base + kSfCol0 + s * kSfColsPerStage;
                tmem_st_16cols(col, va);
                tmem_st_16cols(col + 16, vb);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sf_full[s]);
            }
        }
    } else {
        // ---- epilogue warps: lane quadrant warp & 3 of the accumulator
        const int qe = warp & 3;
        int it = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
            const int tm = t % ntm, tn = t / ntm, b = it & 1;
            if (*abort_flag || !mbar_wait(&acc_full[b], (it >> 1) & 1)) {
                fail();
                break;
            }
            tc_fence_after();
            const int m = tm * kBM + 32 * qe + lane;
#pragma unroll 1
            for (int c = 0; c < kBN; c += 32) {
                // 1/g of token c + lane of the chunk, broadcast per column
                const int nl = tn * kBN + c + lane;
                const float rg = nl < N ? __frcp_rn(__ldg(g + nl)) : 0.0f;
                uint32_t r[32];
                tmem_ld_32cols(tmem + ((uint32_t)(32 * qe) << 16) + b * kAccCols + c, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int n = tn * kBN + c + j;
                    const float f = __shfl_sync(0xffffffffu, rg, j);
                    if (n < N && m < M) Y[(size_t)n * M + m] = __uint_as_float(r[j]) * f;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[b]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kNvTmemCols);
}

}  // namespace

size_t nv_workspace_bytes(int64_t N, int64_t K) {
    const size_t codes = ((size_t)N * K / 2 + 255) / 256 * 256;
    const size_t sf = ((size_t)N * K / 16 + 255) / 256 * 256;
    return codes + sf + (size_t)N * 4;
}

}  // namespace rfp2

using namespace rfp2;

extern "C" size_t rfp2_nvfp4_weight_bytes(int64_t M, int64_t K) {
    if (M <= 0 || K <= 0 || K % 32) return 0;
    return (size_t)M * K / 2 + (size_t)M * K / 16;
}

extern "C" rfp2_status rfp2_to_nvfp4(const uint8_t *W, int64_t M, int64_t K, uint8_t *Wnv,
                                     rfp2_stream_t stream) {
    if (!W || !Wnv) return RFP2_EINVAL;
    if (M <= 0 || K <= 0 || K % 32) return RFP2_ESHAPE;
    if (!aligned(W, 2) || !aligned(Wnv, 16)) return RFP2_EALIGN;
    const int64_t nblocks = M * (K / 32);
    const int threads = 256;
    nv_convert_kernel<<<(unsigned)((nblocks + threads - 1) / threads), threads, 0,
                        reinterpret_cast<cudaStream_t>(stream)>>>(W, nblocks, K / 32, Wnv,
                                                                  Wnv + (size_t)M * K / 2);
    return from_cuda(launch_status());
}

extern "C" size_t rfp2_gemm_nvfp4_workspace_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0) return 0;
    return nv_workspace_bytes(N, K);
}

extern "C" rfp2_status rfp2_gemm_nvfp4(const uint8_t *Wnv, int64_t M, int64_t K, const uint16_t *X,
                                       int64_t N, float *Y, void *workspace, size_t workspace_bytes,
                                       int32_t *dev_status, rfp2_stream_t stream) {
    if (!Wnv || !X || !Y) return RFP2_EINVAL;
    if (M <= 0 || K <= 0 || N <= 0 || M > (1LL << 30) || N > (1LL << 30)) return RFP2_ESHAPE;
    if (K % 256 != 0 || K > (1LL << 24)) return RFP2_EUNSUPPORTED;
    if (!workspace || workspace_bytes < nv_workspace_bytes(N, K)) return RFP2_EWORKSPACE;
    if (!aligned(Wnv, 16) || !aligned(X, 16) || !aligned(Y, 4) || !aligned(workspace, 256))
        return RFP2_EALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *xc = static_cast<uint8_t *>(workspace);
    uint8_t *xs = xc + ((size_t)N * K / 2 + 255) / 256 * 256;
    float *g = reinterpret_cast<float *>(xs + ((size_t)N * K / 16 + 255) / 256 * 256);
    nv_quant_kernel<<<(unsigned)N, kQThreads, 0, s>>>(X, (int)K, xc, xs, g);
    if (launch_status() != cudaSuccess) return RFP2_ECUDA;
    const uint8_t *wsf = Wnv + (size_t)M * K / 2;
    CUtensorMap wmap, xmap, wsmap, xsmap;
    if (!encode_tensor_map_2d(&wmap, Wnv, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)K / 2,
                              (uint64_t)M, (uint64_t)K / 2, kBKB, kBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_2d(&xmap, xc, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)K / 2,
                              (uint64_t)N, (uint64_t)K / 2, kBKB, kBN, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_2d(&wsmap, wsf, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)K / 16,
                              (uint64_t)M, (uint64_t)K / 16, 16, kBM) ||
        !encode_tensor_map_2d(&xsmap, xs, CU_TENSOR_MAP_DATA_TYPE_UINT8, (uint64_t)K / 16,
                              (uint64_t)N, (uint64_t)K / 16, 16, kBN))
        return RFP2_ECUDA;
    static std::mutex mu;
    static int configured[64] = {0};
    const int dev = current_device();
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && configured[dev] == 0) {
            if (set_smem_limit(nv_gemm_kernel, (int)kNvSmem) != cudaSuccess) return RFP2_ECUDA;
            configured[dev] = 1;
        }
    }
    const int64_t ntiles = ((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
    const int sms = sm_count(dev);
    const int grid = (int)(ntiles < sms ? ntiles : sms);
    return from_cuda(launch(nv_gemm_kernel, dim3(grid), dim3(kNvThreads), kNvSmem, s, true, wmap,
                            xmap, wsmap, xsmap, static_cast<const float *>(g), Y, (int)M, (int)N,
                            (int)K, dev_status));
}
