// Dense ROCmFP2 GEMV: y[n, m] = sum_k w[m, k] * q[n, k] * dA (int8 path).
//
// Source: "ROCmFP2 codebook research report", sections "01 Storage",
// "02 Quantization" and "03 Runtime" (LOAD -> SPREAD -> PERMUTE -> DOT4 ->
// RESCALE, with each block expanded once for every activation column).
//
// GB300 design.  The packed weights (2.5 bits per weight) are the only large
// stream, so the kernel is built around HBM:
//  * Persistent grid, one CTA per SM; CTA i owns the contiguous rows
//    [i*M/G, (i+1)*M/G), so its weights are one contiguous slab.
//  * A producer warp streams that slab into a ring of shared-memory stages
//    with 1-D bulk async copies (cp.async.bulk, L2 evict-first), one stage per
//    chunk of rows, issuing as many stages as fit (~200 KB, ~100 KB when two
//    CTAs share the SM) before the first
//    one is consumed.  Rows of K % 256 == 0 are whole 16-byte units.
//  * Batches of at most two quantize x inside the kernel (one launch per
//    call; every CTA quantizes the whole vector into shared memory) and are
//    built to run two CTAs per SM: the next call's CTA becomes resident at
//    once and streams its weights while this call computes.
//  * Twelve or sixteen consumer warps.  Each thread keeps the int8 activations of its
//    K-slice for all N columns in registers, reads its BPT blocks of a row
//    with conflict-free shared loads (strides 20/40/80 B map to distinct
//    banks) and runs the PRMT + dp4a decode of rfp2_decode.cuh.
//  * Every wait is an mbarrier wait with a time limit; a timeout stores
//    RFP2_ETIMEOUT and the CTA winds down after its copies have landed.  The
//    cross-warp reduction (when a row spans several warps) also goes through
//    mbarriers, never through bar.sync, so no wait can hang.
#include <mutex>

#include <algorithm>

#include "common.cuh"
#include "gemv_core.cuh"
#include "quantize.cuh"

namespace rfp2 {
namespace {

// Consumer warps per CTA (+ 1 producer warp).  Batch 1 needs about 70
// registers per thread, so 16 consumer warps fit (the 544-thread block is
// capped at 96 registers); wider batches hold more activations and use 12
// (416 threads, 128 registers).
#ifndef RFP2_GEMV_WARPS1
#define RFP2_GEMV_WARPS1 16
#endif
#ifndef RFP2_GEMV_WARPS
#define RFP2_GEMV_WARPS 12
#endif
// The fused-quantize kernel (batch <= 2): consumer warps, CTAs per SM it is
// compiled for, and its shared-memory budget.  Two CTAs per SM let the next
// call's CTA start beside the running one and prefetch its weights while this
// one computes.
#ifndef RFP2_GEMV_FWARPS
#define RFP2_GEMV_FWARPS 16
#endif
#ifndef RFP2_GEMV_FMINB
#define RFP2_GEMV_FMINB 2
#endif
#ifndef RFP2_GEMV_FUSED_SMEM
#define RFP2_GEMV_FUSED_SMEM (100 * 1024)
#endif
#ifndef RFP2_GEMV_MAX_STAGES
#define RFP2_GEMV_MAX_STAGES 64
#endif
template <int NC, bool FQ>
constexpr int consumer_warps() {
    return FQ ? RFP2_GEMV_FWARPS : NC == 1 ? RFP2_GEMV_WARPS1 : RFP2_GEMV_WARPS;
}
template <int NC, bool FQ>
constexpr int gemv_threads() {
    return (consumer_warps<NC, FQ>() + 1) * 32;
}

// Rows per warp per chunk: several independent rows per warp amortise the
// per-chunk wait, reduction and bookkeeping; capped so R*NC <= 8.
#ifndef RFP2_GEMV_R1
#define RFP2_GEMV_R1 2
#endif
template <int NC>
constexpr int rows_per_warp() {
    return NC == 1 ? RFP2_GEMV_R1 : NC == 2 ? 2 : 1;
}

// FQ = false: q/d come quantized from global memory (copied to shared memory
// by the producer warp).  FQ = true: the consumer warps quantize x into shared
// memory themselves (one launch per call; CTA 0 also writes q/d to global).
template <int NC, int BPT, bool FQ>
__global__ void __launch_bounds__(gemv_threads<NC, FQ>(), FQ ? RFP2_GEMV_FMINB : 1)
    gemv_q8_kernel(const uint8_t *__restrict__ W, int M, int K, const int8_t *__restrict__ q,
                   const float *__restrict__ d, const float *__restrict__ x, int8_t *qout,
                   float *dout, float *__restrict__ y, int32_t *status, int WK, int stages,
                   int rows_per_cta, int rows_extra) {
    extern __shared__ __align__(128) uint8_t smem[];
#ifndef RFP2_GEMV_NO_EARLY_TRIGGER
    // fused path: let the next call's grid become resident at once (beside
    // this CTA) so that its weight stream overlaps this call's compute; its
    // consumers still wait for this grid to complete before touching x or y
    if constexpr (FQ) pdl_launch_dependents();
#endif
    const int KB = K >> 5;
    const int rowbytes = KB * 10;
    constexpr int R = rows_per_warp<NC>();
    constexpr int CW = consumer_warps<NC, FQ>();
    const int RG = CW / WK;  // row groups; R rows per group per chunk
    const int CR = RG * R;   // rows per chunk
    Ring r = carve_ring(smem, stages, CR * rowbytes, RG, WK, NextPow2<R * NC>::v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // CTA i owns rows_per_cta (+1 for the first rows_extra CTAs) contiguous rows
    const int bx = blockIdx.x;
    const int64_t r_begin = (int64_t)bx * rows_per_cta + min(bx, rows_extra);
    const int nrows = rows_per_cta + (bx < rows_extra ? 1 : 0);
    const int64_t r_end = r_begin + nrows;
    const int nchunks = (nrows + CR - 1) / CR;
    const uint8_t *src = W + r_begin * rowbytes;
    const bool producer = warp == CW && lane == 0;
    uint64_t pol = 0;
    int c = 0;
    // activations staged after the ring: q [NC, K] int8 then d [NC, K/32] fp32
    const uint32_t qbytes = (uint32_t)NC * K, dbytes = (uint32_t)NC * KB * 4;
    uint8_t *act_q = smem + ring_bytes(stages, CR * rowbytes, RG, WK, NextPow2<R * NC>::v);
    uint8_t *act_d = act_q + ((qbytes + 15) & ~15u);
    if (producer) {
        // start the weight stream before anything else: the stage barriers
        // are initialised and the first stages issued ahead of the CTA barrier
        init_ring_stages(r, CW, FQ ? CW * 32 : 32);
        pol = policy_evict_first();
        for (; c < nchunks && c < stages; ++c) {
            const int rows = min(CR, nrows - c * CR);
            produce_chunk(r, c, src + (int64_t)c * CR * rowbytes, (uint32_t)(rows * rowbytes), pol,
                          status);
        }
    }
    init_ring_reduction(r, threadIdx.x, CW * 32);
    __syncthreads();

    if (warp == CW) {
        if constexpr (!FQ) {
            // q and d may come from the kernel launched just before this one
            pdl_wait();
            load_act_to_smem(r, lane, act_q, q, qbytes, act_d, d, dbytes);
        }
        // producer: refill the ring as the consumers release stages
        if (lane == 0) {
            for (; c < nchunks; ++c) {
                const int rows = min(CR, nrows - c * CR);
                if (!produce_chunk(r, c, src + (int64_t)c * CR * rowbytes,
                                   (uint32_t)(rows * rowbytes), pol, status))
                    break;
            }
            drain_ring(r, c, status);
        }
        return;
    }

    const int wg = warp / WK, wk = warp % WK;
    const int kb0 = (wk * 32 + lane) * BPT;
    const bool active = kb0 < KB;
    pdl_wait();
    pdl_launch_dependents();
    if constexpr (FQ)
        quantize_to_smem(r, warp, CW, lane, x, NC, K, act_q, reinterpret_cast<float *>(act_d),
                         blockIdx.x == 0 ? qout : nullptr, dout);
    if (!mbar_wait(r.act_bar, 0)) {
        record_status(status, RFP2_ETIMEOUT);
        *r.abort_flag = 1;
        return;
    }
    Act<NC, BPT> A;
    int cols[NC];
    float *ycol[NC];
#pragma unroll
    for (int n = 0; n < NC; ++n) {
        cols[n] = n;
        ycol[n] = y + (int64_t)n * M;
    }
    load_act<NC, BPT, true>(A, reinterpret_cast<const int8_t *>(act_q),
                      reinterpret_cast<const float *>(act_d), K, kb0, active, cols);
    for (c = 0; c < nchunks; ++c) {
        int64_t rows[R];
        bool valid[R];
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            rows[rr] = r_begin + (int64_t)c * CR + wg * R + rr;
            valid[rr] = rows[rr] < r_end;
        }
        if (!consume_chunk<NC, BPT, R>(r, c, wg, wk, lane, kb0, active, rowbytes, rows, valid, A,
                                       ycol, status))
            break;
    }
}

// ---------------------------------------------------------------------------
// Host side

struct Plan {
    int bpt, WK, RG, chunk_bytes, stages, grid;
    size_t smem;
};

bool make_plan(int NC, int64_t M, int64_t K, Plan &p, bool fused = false) {
    const size_t budget = fused ? (size_t)RFP2_GEMV_FUSED_SMEM : (size_t)kGemvSmemBudget;
    const int KB = (int)(K / 32);
    int bpt = bpt_max(NC);
    while (bpt > 1 && KB < 32 * bpt) bpt /= 2;
    int WK = (KB + 32 * bpt - 1) / (32 * bpt);
    // K-slice warps per row: the smallest divisor of the consumer warp count
    // that covers the row (row groups of CW / WK warps)
    const int CW = fused ? consumer_warps<1, true>()
                   : NC == 1 ? consumer_warps<1, false>() : consumer_warps<2, false>();
    int WKp = 0;
    for (int dv = 1; dv <= CW; ++dv)
        if (CW % dv == 0 && dv >= WK) {
            WKp = dv;
            break;
        }
    if (WKp == 0) return false;
    p.bpt = bpt;
    p.WK = WKp;
    p.RG = CW / WKp;
    const int R = NC == 1 ? rows_per_warp<1>() : NC == 2 ? rows_per_warp<2>() : 1;
    const int CR = p.RG * R;
    const int rowbytes = KB * 10;
    p.chunk_bytes = CR * rowbytes;
    const int64_t chunks_total = (M + CR - 1) / CR;
    const int sms = sm_count(current_device());
    p.grid = (int)(chunks_total < sms ? chunks_total : sms);
    const int64_t rows_per_cta = (M + p.grid - 1) / p.grid;
    const int chunks_per_cta = (int)((rows_per_cta + CR - 1) / CR);
    const int RN = R * NC;
    const int V = RN <= 1 ? 1 : RN <= 2 ? 2 : RN <= 4 ? 4 : 8;
    const size_t act = ((size_t)NC * K + 15) / 16 * 16 + (size_t)NC * KB * 4;
    int stages = chunks_per_cta < RFP2_GEMV_MAX_STAGES ? chunks_per_cta : RFP2_GEMV_MAX_STAGES;
    while (stages > 1 &&
           ring_bytes(stages, p.chunk_bytes, p.RG, p.WK, V) + act > budget)
        --stages;
    p.stages = stages;
    p.smem = ring_bytes(stages, p.chunk_bytes, p.RG, p.WK, V) + act;
    return p.smem <= 227 * 1024;
}

template <int NC, int BPT, bool FQ>
cudaError_t launch_gemv_t(const Plan &p, const uint8_t *W, int M, int K, const int8_t *q,
                          const float *d, const float *x, int8_t *qout, float *dout, float *y,
                          int32_t *status, cudaStream_t stream, bool pdl) {
    auto kern = gemv_q8_kernel<NC, BPT, FQ>;
    static std::mutex mu;
    static int configured[64] = {0};
    const int dev = current_device();
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && configured[dev] == 0) {
            cudaError_t e = set_smem_limit(kern, 227 * 1024);
            if (e != cudaSuccess) return e;
            configured[dev] = 1;
        }
    }
    return launch(kern, dim3(p.grid), dim3(gemv_threads<NC, FQ>()), p.smem, stream, pdl, W, M, K,
                  q, d, x, qout, dout, y, status, p.WK, p.stages, M / p.grid, M % p.grid);
}

template <int NC, bool FQ>
cudaError_t launch_gemv_nc(const Plan &p, const uint8_t *W, int M, int K, const int8_t *q,
                           const float *d, const float *x, int8_t *qout, float *dout, float *y,
                           int32_t *status, cudaStream_t stream, bool pdl) {
    switch (p.bpt) {
        case 8:
            if constexpr (bpt_max(NC) >= 8)
                return launch_gemv_t<NC, 8, FQ>(p, W, M, K, q, d, x, qout, dout, y, status, stream,
                                                pdl);
            break;
        case 4:
            if constexpr (bpt_max(NC) >= 4)
                return launch_gemv_t<NC, 4, FQ>(p, W, M, K, q, d, x, qout, dout, y, status, stream,
                                                pdl);
            break;
        case 2:
            if constexpr (bpt_max(NC) >= 2)
                return launch_gemv_t<NC, 2, FQ>(p, W, M, K, q, d, x, qout, dout, y, status, stream,
                                                pdl);
            break;
        default:
            return launch_gemv_t<NC, 1, FQ>(p, W, M, K, q, d, x, qout, dout, y, status, stream, pdl);
    }
    return cudaErrorInvalidValue;
}

// GEMV on quantized activations q/d.
cudaError_t launch_gemv(const uint8_t *W, int64_t M, int64_t K, const int8_t *q, const float *d,
                        int64_t N, float *y, int32_t *status, cudaStream_t stream, bool pdl) {
    Plan p;
    if (!make_plan((int)N, M, K, p)) return cudaErrorInvalidValue;
    const int m = (int)M, k = (int)K;
    switch (N) {
#define RFP2_CASE(n)                                                                            \
    case n:                                                                                     \
        return launch_gemv_nc<n, false>(p, W, m, k, q, d, nullptr, nullptr, nullptr, y, status, \
                                        stream, pdl);
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

// Batches of at most 2 whose activations fit beside a weight ring: quantize
// inside the GEMV (one launch per call); q and d also go to qout/dout.
bool fused_applies(int64_t M, int64_t K, int64_t N) {
    Plan p;
    return N <= 2 && make_plan((int)N, M, K, p, true);
}

cudaError_t launch_gemv_fused(const uint8_t *W, int64_t M, int64_t K, const float *x, int64_t N,
                              int8_t *qout, float *dout, float *y, int32_t *status,
                              cudaStream_t stream) {
    Plan p;
    if (!make_plan((int)N, M, K, p, true)) return cudaErrorInvalidValue;
    const int m = (int)M, k = (int)K;
    if (N == 1)
        return launch_gemv_nc<1, true>(p, W, m, k, nullptr, nullptr, x, qout, dout, y, status,
                                       stream, true);
    return launch_gemv_nc<2, true>(p, W, m, k, nullptr, nullptr, x, qout, dout, y, status, stream,
                                   true);
}

rfp2_status check_gemv_shape(int64_t M, int64_t K, int64_t N) {
    if (M <= 0 || K <= 0 || N < 1 || N > RFP2_MAX_BATCH) return RFP2_ESHAPE;
    if (M > (1LL << 30) || K > (1LL << 30)) return RFP2_ESHAPE;
    if (K % 256 != 0) return RFP2_EUNSUPPORTED;
    Plan p;
    if (!make_plan((int)N, M, K, p)) return RFP2_EUNSUPPORTED;
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
    const rfp2_status st = check_gemv_shape(M, K, N);
    if (st != RFP2_OK) return st;
    if (!aligned(W, 16) || !aligned(q, 16) || !aligned(d, 16) || !aligned(y, 4)) return RFP2_EALIGN;
    return from_cuda(launch_gemv(W, M, K, q, d, N, y, dev_status,
                                 reinterpret_cast<cudaStream_t>(stream), false));
}

// From three tokens on, the tensor-core verify-batch path (decode straight
// into tensor memory, ~18 us for the 14336 x 4096 decode weights at any N up
// to 32) beats the dp4a GEMV (19.6 us at N = 3, 44 us at N = 8); both give the
// int path's result within the 1e-5 bar.  It needs M % 16 == 0 and x 16-byte
// aligned; its workspace starts with the same q and d.
static bool use_tensor_path(int64_t M, int64_t N, const void *x) {
    return N >= 3 && M % 16 == 0 && (x == nullptr || rfp2::aligned(x, 16));
}

extern "C" size_t rfp2_gemv_workspace_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0) return 0;
    size_t b = gemv_workspace_bytes(N, K);
    if (N >= 3) b = std::max(b, rfp2_gemv_batched_workspace_bytes(16, K, N));
    return b;
}

extern "C" rfp2_status rfp2_gemv(const uint8_t *W, int64_t M, int64_t K, const float *x,
                                 int64_t N, float *y, void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, rfp2_stream_t stream) {
    if (!W || !x || !y) return RFP2_EINVAL;
    if (M <= 0 || K <= 0 || N < 1 || N > RFP2_MAX_BATCH) return RFP2_ESHAPE;
    // the tensor path has its own limits (no activation staging beside a ring)
    if (K % 256 == 0 && use_tensor_path(M, N, x))
        return rfp2_gemv_batched(W, M, K, x, N, y, workspace, workspace_bytes, dev_status, stream);
    const rfp2_status st = check_gemv_shape(M, K, N);
    if (st != RFP2_OK) return st;
    if (!workspace || workspace_bytes < gemv_workspace_bytes(N, K)) return RFP2_EWORKSPACE;
    if (!aligned(W, 16) || !aligned(x, 4) || !aligned(y, 4) || !aligned(workspace, 256))
        return RFP2_EALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int8_t *q = static_cast<int8_t *>(workspace);
    float *d = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                         ((size_t)(N * K) + 255) / 256 * 256);
    if (fused_applies(M, K, N))
        return from_cuda(launch_gemv_fused(W, M, K, x, N, q, d, y, dev_status, s));
    cudaError_t e = launch_quantize(x, N, K, q, d, s, true);
    if (e != cudaSuccess) return RFP2_ECUDA;
    return from_cuda(launch_gemv(W, M, K, q, d, N, y, dev_status, s, true));
}

// ---------------------------------------------------------------------------
// rfp2_gemv_noalloc: rfp2_gemv for callers that cannot allocate device
// memory.  Some callers run where a cudaMalloc is not allowed or not
// possible: a plugin inside another runtime that owns the device memory
// pool, code running under a memory budget that must not grow, or a path that
// has to work after the pool is exhausted.  For them the quantized
// activations (the only scratch rfp2_gemv needs) live in a fixed array in
// device global memory that belongs to the library: every GPU that loads the
// library holds it until the process exits.  The array is shared by every
// call on a device, so calls that overlap on the GPU (different streams,
// different host threads) race on it and must be serialized by the caller.
// Nothing in it needs to start at zero: each call overwrites the part it uses.

namespace rfp2 {
namespace {

// q int8 [N, K] (N*K <= kNoAllocMaxNK bytes) followed by d fp32 [N, K/32].
constexpr int64_t kNoAllocMaxNK = 65536;
constexpr size_t kNoAllocQBytes = kNoAllocMaxNK;
constexpr size_t kNoAllocBytes = kNoAllocQBytes + kNoAllocMaxNK / 32 * sizeof(float);
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];

// Device address of the array, looked up once per device with that device
// current (in host code the array's name is only a host-side stand-in).
uint8_t *noalloc_scratch_ptr(int dev, cudaError_t *err) {
    static std::mutex mu;
    static uint8_t *ptrs[64] = {nullptr};
    if (dev < 0 || dev >= 64) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) {
            *err = e;
            return nullptr;
        }
        ptrs[dev] = static_cast<uint8_t *>(p);
    }
    *err = cudaSuccess;
    return ptrs[dev];
}

}  // namespace
}  // namespace rfp2

extern "C" rfp2_status rfp2_gemv_noalloc(const uint8_t *W, int64_t M, int64_t K, const float *x,
                                         int64_t N, float *y, int32_t *dev_status,
                                         rfp2_stream_t stream) {
    if (!W || !x || !y) return RFP2_EINVAL;
    if (M <= 0 || K <= 0 || N < 1 || N > RFP2_MAX_BATCH) return RFP2_ESHAPE;
    if (N * K > kNoAllocMaxNK) return RFP2_EWORKSPACE;  // beyond the built-in scratch
    const rfp2_status st = check_gemv_shape(M, K, N);
    if (st != RFP2_OK) return st;
    if (!aligned(W, 16) || !aligned(x, 4) || !aligned(y, 4)) return RFP2_EALIGN;
    cudaError_t e = cudaSuccess;
    uint8_t *scratch = noalloc_scratch_ptr(current_device(), &e);
    if (!scratch) return RFP2_ECUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int8_t *q = reinterpret_cast<int8_t *>(scratch);
    float *d = reinterpret_cast<float *>(scratch + kNoAllocQBytes);
    e = launch_quantize(x, N, K, q, d, s, true);
    if (e != cudaSuccess) return RFP2_ECUDA;
    return from_cuda(launch_gemv(W, M, K, q, d, N, y, dev_status, s, true));
}
