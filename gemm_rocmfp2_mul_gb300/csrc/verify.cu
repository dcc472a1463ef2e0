// ROCmFP2 GEMV for verify batches (tens to hundreds of tokens) on the
// 5th-generation tensor cores, with the results of the Q8_1 int path:
// y[n, m] = sum_b dA[n, b] * sum_{k in b} w[m, k] * q[n, k].
//
// Source: "ROCmFP2 codebook research report", section "03 Runtime" (Q8_1
// activations; expand each block once and reuse it for every activation
// column, the mid-range between the GEMV and the GEMM).
//
// Four launches chained with programmatic dependent launch:
//  1. expand: packed blocks -> f16 weights (exact) in the workspace;
//  2. quantize the tokens (Q8_1 blocks, the same kernel as rfp2_gemv);
//  3. split: x^ = q * dA scaled by 2^-kc (per token) into two f16 pieces,
//     hi + lo, relative residual <= 2^-22;
//  4. vb_gemm: one CTA per 128 weight rows x BNT tokens.  Warp 0 streams
//     K-major 64-element slices of the weights and of both activation pieces
//     with 2-D TMA (SWIZZLE_128B) into a ring; one thread of warp 1 issues
//     tcgen05.mma kind::f16 (M = 128 weight rows, N = BNT tokens, K = 16,
//     f16 in, fp32 in tensor memory).  The tensor cores' fp32 accumulation
//     does not round to nearest, which over 2K/16 steps would cost ~1.5e-5
//     relative; so the product is accumulated in short chunks (16 MMAs)
//     in two alternating tensor-memory buffers, and warps 2-5 add each
//     finished chunk into fp32 registers (one weight row per thread, BNT
//     token sums) while the next chunk runs.  They then store y with 2^kc.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "expand.cuh"
#include "quantize.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace rfp2 {
namespace {

constexpr int VBM = 128;      // weight rows per tile (UMMA M)
constexpr int VBK = 64;       // K per stage: one 128-byte swizzle row of f16
constexpr int VUK = 16;       // K per UMMA instruction
constexpr int VSTAGES = 4;
constexpr int VCHUNK = 2;     // stages (2 x 8 MMAs) per tensor-memory accumulation chunk
constexpr int VTHREADS = 6 * 32;
constexpr int kABytes = VBM * VBK * 2;

// one stage: the weight slice and both activation pieces of the same K range
template <int BNT>
constexpr int stage_bytes() { return kABytes + 2 * BNT * VBK * 2; }
template <int BNT>
constexpr size_t vb_smem_bytes() { return 1024 + (size_t)VSTAGES * stage_bytes<BNT>() + 256; }

// x^ = q * dA of token n as two f16 pieces after an exact power-of-two
// scaling (kc from max 127 * dA, so every scaled value is below 2).  Grid
// (slices, N); every CTA of a token reads its K/32 scales and writes one
// slice of hi and lo, row-major [N, K].
__global__ void __launch_bounds__(256) vb_split_kernel(const int8_t *__restrict__ q,
                                                       const float *__restrict__ d, int N, int K,
                                                       __half *__restrict__ xhi,
                                                       __half *__restrict__ xlo, int *kc_out) {
    __shared__ float wmax[8];
    pdl_wait();
    pdl_launch_dependents();
    const int n = blockIdx.y;
    const int KB = K >> 5;
    const float *dr = d + (int64_t)n * KB;
    float dmax = 0.0f;
    for (int b = threadIdx.x; b < KB; b += blockDim.x) dmax = fmaxf(dmax, dr[b]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        dmax = fmaxf(dmax, __shfl_xor_sync(0xffffffffu, dmax, off));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = dmax;
    __syncthreads();
    dmax = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) dmax = fmaxf(dmax, wmax[i]);
    const float bound = 127.0f * dmax;  // >= max |q * dA| of the token
    const int kc = bound > 0.0f ? ilogbf(bound) : 0;
    if (threadIdx.x == 0 && blockIdx.x == 0) kc_out[n] = kc;
    const int per = (K + gridDim.x - 1) / gridDim.x;
    const int k0 = blockIdx.x * per, k1 = min(K, k0 + per);
    const int8_t *qr = q + (int64_t)n * K;
    for (int k = k0 + threadIdx.x; k < k1; k += blockDim.x) {
        const float v = ldexpf((float)qr[k] * dr[k >> 5], -kc);
        const __half h = __float2half_rn(v);
        xhi[(int64_t)n * K + k] = h;
        xlo[(int64_t)n * K + k] = __float2half_rn(v - __half2float(h));
    }
}

template <int BNT>
__global__ void __launch_bounds__(VTHREADS, 1)
    vb_gemm_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap hmap,
                   const __grid_constant__ CUtensorMap lmap, float *__restrict__ y, int Mw,
                   int Ntok, int K, const int *__restrict__ kc, int32_t *status) {
    constexpr int SB = stage_bytes<BNT>();
    constexpr uint32_t kTmemCols = 2 * BNT < 32 ? 32 : 2 * BNT;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)VSTAGES * SB);
    uint64_t *empty = full + VSTAGES;
    uint64_t *accf = empty + VSTAGES;  // [2] chunk finished in buffer b
    uint64_t *acce = accf + 2;         // [2] buffer b read back
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acce + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile_m = blockIdx.x, tile_n = blockIdx.y;
    const int nk = K / VBK;
    const int nt = nk;
    const int nchunks = (nt + VCHUNK - 1) / VCHUNK;
    constexpr int kBBytes = BNT * VBK * 2;

    if (threadIdx.x == 0) {
        prefetch_tensor_map(&wmap);
        prefetch_tensor_map(&hmap);
        prefetch_tensor_map(&lmap);
        for (int s = 0; s < VSTAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 4);  // one arrival per epilogue warp
        }
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

    if (warp == 0 && lane == 0) {
        // ---- TMA producer: weights (A) and one activation piece (B) per slice
        pdl_wait();
        int t = 0;
        for (; t < nt; ++t) {
            const int s = t % VSTAGES;
            if (t >= VSTAGES && !mbar_wait(&empty[s], ((t / VSTAGES) - 1) & 1)) {
                record_status(status, RFP2_ETIMEOUT);
                *abort_flag = 1;
                break;
            }
            if (*abort_flag) break;
            uint8_t *a = smem + (size_t)s * SB;
            mbar_arrive_expect_tx(&full[s], SB);
            tma_load_2d(a, &wmap, t * VBK, tile_m * VBM, &full[s]);
            tma_load_2d(a + kABytes, &hmap, t * VBK, tile_n * BNT, &full[s]);
            tma_load_2d(a + kABytes + kBBytes, &lmap, t * VBK, tile_n * BNT, &full[s]);
        }
        for (int i = max(0, t - VSTAGES); i < t; ++i)
            if (!mbar_wait(&full[i % VSTAGES], (i / VSTAGES) & 1))
                record_status(status, RFP2_ETIMEOUT);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer: chunk c accumulates into buffer c & 1
        constexpr uint32_t idesc = idesc_f16_f32(VBM, BNT);
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            const int b = c & 1;
            if (c >= 2 && (*abort_flag || !mbar_wait(&acce[b], ((c >> 1) - 1) & 1))) {
                record_status(status, RFP2_ETIMEOUT);
                *abort_flag = 1;
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + (uint32_t)(b * BNT);
            const int t0 = c * VCHUNK, t1 = min(nt, t0 + VCHUNK);
            for (int t = t0; t < t1; ++t) {
                const int s = t % VSTAGES;
                if (*abort_flag || !mbar_wait(&full[s], (t / VSTAGES) & 1)) {
                    record_status(status, RFP2_ETIMEOUT);
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a = smem_addr(smem + (size_t)s * SB);
                const uint64_t adesc = smem_desc_sw128(a);
#pragma unroll
                for (int piece = 0; piece < 2; ++piece) {
                    const uint64_t bdesc = smem_desc_sw128(a + kABytes + piece * kBBytes);
#pragma unroll
                    for (int k = 0; k < VBK / VUK; ++k)
                        umma_bf16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc,
                                  (t > t0 || piece > 0 || k > 0) ? 1u : 0u);
                }
                umma_commit(&empty[s]);
            }
            umma_commit(&accf[b]);  // chunk complete (or, after an abort, idle)
        }
    } else if (warp >= 2) {
        // ---- epilogue: add every finished chunk into fp32 registers
        const int q = warp & 3;  // tensor-memory lanes 32q .. 32q+31 = weight rows
        const int m = tile_m * VBM + q * 32 + lane;
        float acc[BNT];
#pragma unroll
        for (int i = 0; i < BNT; ++i) acc[i] = 0.0f;
        bool ok = true;
        for (int c = 0; c < nchunks; ++c) {
            const int b = c & 1;
            if (*abort_flag || !mbar_wait(&accf[b], (c >> 1) & 1)) {
                record_status(status, RFP2_ETIMEOUT);
                *abort_flag = 1;
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < BNT / 32; ++j) {
                uint32_t r[32];
                tmem_ld_32cols(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BNT + j * 32), r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) acc[j * 32 + i] += __uint_as_float(r[i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[b]);
        }
        if (ok && m < Mw) {
#pragma unroll
            for (int i = 0; i < BNT; ++i) {
                const int n = tile_n * BNT + i;
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
    __half *wexp;
    int8_t *q;
    float *d;
    __half *xhi, *xlo;
    int *kc;
    size_t bytes;
};

VbWs carve_vb(void *ws, int64_t M, int64_t K, int64_t N) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    uint8_t *p = static_cast<uint8_t *>(ws);
    VbWs w;
    size_t o = 0;
    w.wexp = reinterpret_cast<__half *>(p + o);
    o += up((size_t)M * K * 2);
    w.q = reinterpret_cast<int8_t *>(p + o);
    o += up((size_t)N * K);
    w.d = reinterpret_cast<float *>(p + o);
    o += up((size_t)N * (K / 32) * 4);
    w.xhi = reinterpret_cast<__half *>(p + o);
    o += up((size_t)N * K * 2);
    w.xlo = reinterpret_cast<__half *>(p + o);
    o += up((size_t)N * K * 2);
    w.kc = reinterpret_cast<int *>(p + o);
    o += up((size_t)N * 4);
    w.bytes = o;
    return w;
}

template <int BNT>
cudaError_t launch_vb_gemm(const VbWs &w, float *y, int64_t M, int64_t K, int64_t N,
                           int32_t *status, cudaStream_t s) {
    CUtensorMap wmap, hmap, lmap;
    if (!encode_tensor_map_2d(&wmap, w.wexp, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (uint64_t)K,
                              (uint64_t)M, (uint64_t)K * 2, VBK, VBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_2d(&hmap, w.xhi, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (uint64_t)K,
                              (uint64_t)N, (uint64_t)K * 2, VBK, BNT, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_2d(&lmap, w.xlo, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (uint64_t)K,
                              (uint64_t)N, (uint64_t)K * 2, VBK, BNT, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    static std::mutex mu;
    static int configured[64] = {0};
    const int dev = current_device();
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && !configured[dev]) {
            cudaError_t e = set_smem_limit(vb_gemm_kernel<BNT>, (int)vb_smem_bytes<BNT>());
            if (e != cudaSuccess) return e;
            configured[dev] = 1;
        }
    }
    const dim3 grid((unsigned)((M + VBM - 1) / VBM), (unsigned)((N + BNT - 1) / BNT));
    return launch(vb_gemm_kernel<BNT>, grid, dim3(VTHREADS), vb_smem_bytes<BNT>(), s, true, wmap,
                  hmap, lmap, y, (int)M, (int)N, (int)K, static_cast<const int *>(w.kc), status);
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
    if (!aligned(W, 16) || !aligned(x, 4) || !aligned(y, 4) || !aligned(workspace, 256))
        return RFP2_EALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t nblocks = M * (K / 32);
    cudaError_t e = launch(expand_kernel<__half>, dim3((unsigned)((nblocks + 255) / 256)),
                           dim3(256), 0, s, true, W, nblocks, w.wexp);
    if (e != cudaSuccess) return RFP2_ECUDA;
    e = launch_quantize(x, N, K, w.q, w.d, s, true);
    if (e != cudaSuccess) return RFP2_ECUDA;
    const int slices = (int)std::min<int64_t>(32, std::max<int64_t>(1, K / 1024));
    e = launch(vb_split_kernel, dim3((unsigned)slices, (unsigned)N), dim3(256), 0, s, true,
               static_cast<const int8_t *>(w.q), static_cast<const float *>(w.d), (int)N, (int)K,
               w.xhi, w.xlo, w.kc);
    if (e != cudaSuccess) return RFP2_ECUDA;
    if (N <= 32) e = launch_vb_gemm<32>(w, y, M, K, N, dev_status, s);
    else if (N <= 64) e = launch_vb_gemm<64>(w, y, M, K, N, dev_status, s);
    else e = launch_vb_gemm<128>(w, y, M, K, N, dev_status, s);
    return from_cuda(e);
}
