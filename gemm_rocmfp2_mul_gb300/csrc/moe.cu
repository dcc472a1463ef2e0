// MoE bulk-expert GEMV: y[t, j, :] = W[ids[t, j]] x_t for T tokens routed to
// top_k of E ROCmFP2 experts (MUL_MAT_ID run as a GEMV over the routed
// experts' rows for a few tokens: "HRX on the Radeon iGPU", section "MoE
// decode and the kernel cache"; expand-once multi-column reuse: "ROCmFP2
// codebook research report", section "03 Runtime").
//
// Three launches chained with programmatic dependent launch:
//  1. route (one CTA): validates the ids (an id outside [0, E) is never
//     dereferenced: its output row is filled with NaN and RFP2_EBADID is
//     recorded), sorts the (token, slot) pairs by expert and cuts each
//     expert's run into groups of at most 4 pairs.  Groups go to the
//     workspace.
//  2. quantize the T tokens once (Q8_1-style blocks) into the workspace.
//  3. moe_gemv (persistent, one CTA per SM): work units are (group, tile of
//     rows of that expert); CTA i takes a contiguous range of units, its
//     producer warp streams the expert rows into the shared-memory ring and
//     the consumer warps expand every block once for the group's tokens.
//     Expert offsets are 64-bit.
#include <mutex>

#include "common.cuh"
#include "gemv_core.cuh"
#include "quantize.cuh"

namespace rfp2 {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kGemvThreads = (kConsumerWarps + 1) * 32;
constexpr int kGroupCols = 4;        // tokens per group (activation registers)
constexpr int kBpt = 2;              // bpt_max(4)
constexpr int kChunksPerTile = 8;    // rows per unit = 8 chunks of RG rows
constexpr int kMaxPairs = 4096;
constexpr int kRouteThreads = 1024;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct MoeWs {
    int8_t *q;
    float *d;
    int *header;   // [0] groups, [1] valid pairs
    int4 *groups;  // {expert, offset into sorted, ncol, 0}
    int *sorted;   // pair indices p = t * top_k + j sorted by (expert, p)
};

size_t moe_ws_bytes(int64_t T, int64_t top_k, int64_t K) {
    const int64_t P = T * top_k;
    return align256((size_t)(T * K)) + align256((size_t)(T * (K / 32)) * 4) + 256 +
           align256((size_t)P * 16) + align256((size_t)P * 4);
}

MoeWs carve_ws(void *ws, int64_t T, int64_t top_k, int64_t K) {
    uint8_t *p = static_cast<uint8_t *>(ws);
    MoeWs w;
    w.q = reinterpret_cast<int8_t *>(p);
    p += align256((size_t)(T * K));
    w.d = reinterpret_cast<float *>(p);
    p += align256((size_t)(T * (K / 32)) * 4);
    w.header = reinterpret_cast<int *>(p);
    p += 256;
    w.groups = reinterpret_cast<int4 *>(p);
    p += align256((size_t)(T * top_k) * 16);
    w.sorted = reinterpret_cast<int *>(p);
    return w;
}

// Exclusive prefix sum over n <= kMaxPairs flags held in smem, in place.
__device__ void block_exclusive_scan(int *v, int n, int *warp_sums) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int per = kMaxPairs / kRouteThreads;  // 4 per thread
    int local[per];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < per; ++i) {
        const int idx = tid * per + i;
        local[i] = idx < n ? v[idx] : 0;
        sum += local[i];
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int ws = warp_sums[lane];
        int wi = ws;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += t;
        }
        warp_sums[lane] = wi - ws;  // exclusive prefix of warp totals
    }
    __syncthreads();
    int run = warp_sums[warp] + incl - sum;
#pragma unroll
    for (int i = 0; i < per; ++i) {
        const int idx = tid * per + i;
        if (idx < n) v[idx] = run;
        run += local[i];
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kRouteThreads, 1)
    moe_route_kernel(const int32_t *__restrict__ ids, int P, int64_t E, int M, float *y,
                     int32_t *status, MoeWs w) {
    __shared__ int sid[kMaxPairs];         // expert of pair p, -1 if invalid
    __shared__ int gidx[kMaxPairs];        // by sorted position: group-start flag, then index
    __shared__ short left[kMaxPairs];      // by sorted position: pairs left in the expert run
    __shared__ unsigned char flag[kMaxPairs];
    __shared__ int warp_sums[32];
    __shared__ int nvalid_s;
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x;
    if (tid == 0) nvalid_s = 0;
    __syncthreads();
    for (int p = tid; p < P; p += blockDim.x) {
        const int32_t e = ids[p];
        const bool ok = e >= 0 && (int64_t)e < E;
        sid[p] = ok ? e : -1;
        if (!ok) record_status(status, RFP2_EBADID);
        else atomicAdd(&nvalid_s, 1);
    }
    __syncthreads();
    const int nvalid = nvalid_s;
    // NaN rows for invalid pairs (their ids are never used as expert offsets)
    for (int p = 0; p < P; ++p) {
        if (sid[p] >= 0) continue;
        for (int m = tid; m < M; m += blockDim.x) y[(int64_t)p * M + m] = __int_as_float(0x7fc00000);
    }
    // rank of each valid pair by (expert, p), its position inside the
    // expert's run and the run length
    for (int p = tid; p < P; p += blockDim.x) {
        const int e = sid[p];
        if (e < 0) continue;
        int rank = 0, before = 0, count = 0;
        for (int p2 = 0; p2 < P; ++p2) {
            const int e2 = sid[p2];
            if (e2 < 0) continue;
            rank += (e2 < e) || (e2 == e && p2 < p);
            before += e2 < e;
            count += e2 == e;
        }
        const int pos = rank - before;
        w.sorted[rank] = p;
        flag[rank] = (pos % kGroupCols) == 0;
        gidx[rank] = (pos % kGroupCols) == 0;
        left[rank] = (short)(count - pos);
    }
    __syncthreads();
    block_exclusive_scan(gidx, nvalid, warp_sums);  // gidx[r] = starts before r
    for (int r = tid; r < nvalid; r += blockDim.x) {
        if (!flag[r]) continue;
        const int e = sid[w.sorted[r]];
        w.groups[gidx[r]] = make_int4(e, r, min(kGroupCols, (int)left[r]), 0);
    }
    if (tid == 0) {
        w.header[0] = nvalid > 0 ? gidx[nvalid - 1] + flag[nvalid - 1] : 0;
        w.header[1] = nvalid;
    }
}

struct MoeArgs {
    const uint8_t *W;
    int64_t expert_bytes;
    int M, K, T, top_k, WK, nstages, tile_rows;
    int act_staged;  // token activations staged in shared memory
    float *y;
    int32_t *status;
    MoeWs ws;
};

template <int NC>
__device__ bool consume_group(Ring &r, const MoeArgs &a, int4 grp, int t_begin, int t_end, int &c,
                              int wg, int wk, int lane, int kb0, bool active, int rowbytes,
                              const int8_t *q, const float *d, bool staged) {
    int cols[NC];
    float *ycol[NC];
#pragma unroll
    for (int n = 0; n < NC; ++n) {
        const int pair = a.ws.sorted[grp.y + n];
        cols[n] = pair / a.top_k;
        ycol[n] = a.y + (int64_t)pair * a.M;
    }
    Act<NC, kBpt> A;
    if (staged)
        load_act<NC, kBpt, true>(A, q, d, a.K, kb0, active, cols);
    else
        load_act<NC, kBpt, false>(A, q, d, a.K, kb0, active, cols);
    for (int t = t_begin; t < t_end; ++t) {
        const int r0 = t * a.tile_rows;
        const int r1 = min(a.M, r0 + a.tile_rows);
        const int nch = (r1 - r0 + r.RG - 1) / r.RG;
        for (int ch = 0; ch < nch; ++ch, ++c) {
            const int64_t rows[1] = {r0 + (int64_t)ch * r.RG + wg};
            const bool valid[1] = {rows[0] < r1};
            if (!consume_chunk<NC, kBpt, 1>(r, c, wg, wk, lane, kb0, active, rowbytes, rows, valid,
                                            A, ycol, a.status))
                return false;
        }
    }
    return true;
}

__global__ void __launch_bounds__(kGemvThreads, 1) moe_gemv_kernel(MoeArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int KB = a.K >> 5;
    const int rowbytes = KB * 10;
    const int RG = kConsumerWarps / a.WK;
    Ring r = carve_ring(smem, a.nstages, RG * rowbytes, RG, a.WK, NextPow2<kGroupCols>::v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t qbytes = (uint32_t)a.T * a.K, dbytes = (uint32_t)a.T * KB * 4;
    uint8_t *act_q = smem + ring_bytes(a.nstages, RG * rowbytes, RG, a.WK, NextPow2<kGroupCols>::v);
    uint8_t *act_d = act_q + ((qbytes + 15) & ~15u);
    if (threadIdx.x == kConsumerWarps * 32) init_ring_stages(r, kConsumerWarps);
    init_ring_reduction(r, threadIdx.x, kConsumerWarps * 32);
    __syncthreads();
    // the group list and the quantized tokens come from the two launches before
    pdl_wait();
    pdl_launch_dependents();
    if (a.act_staged && warp == kConsumerWarps)
        load_act_to_smem(r, lane, act_q, a.ws.q, qbytes, act_d, a.ws.d, dbytes);
    const int ngroups = a.ws.header[0];
    const int tiles = (a.M + a.tile_rows - 1) / a.tile_rows;
    // units (group, row tile) split into contiguous, balanced CTA ranges
    const int units = ngroups * tiles;
    const int per = units / (int)gridDim.x, extra = units % (int)gridDim.x;
    const int bx = blockIdx.x;
    const int64_t u0 = (int64_t)bx * per + min(bx, extra);
    const int64_t u1 = u0 + per + (bx < extra ? 1 : 0);

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int c = 0;
            bool ok = true;
            for (int64_t u = u0; u < u1 && ok; ++u) {
                const int g = (int)(u / tiles), t = (int)(u % tiles);
                const int4 grp = a.ws.groups[g];
                const uint8_t *base = a.W + (int64_t)grp.x * a.expert_bytes;
                const int r0 = t * a.tile_rows;
                const int r1 = min(a.M, r0 + a.tile_rows);
                for (int row = r0; row < r1 && ok; row += RG, ++c) {
                    const int rows = min(RG, r1 - row);
                    ok = produce_chunk(r, c, base + (int64_t)row * rowbytes,
                                       (uint32_t)(rows * rowbytes), pol, a.status);
                    if (!ok) break;
                }
            }
            drain_ring(r, c, a.status);
        }
        return;
    }

    const int wg = warp / a.WK, wk = warp % a.WK;
    const int kb0 = (wk * 32 + lane) * kBpt;
    const bool active = kb0 < KB;
    const int8_t *q = a.ws.q;
    const float *d = a.ws.d;
    if (a.act_staged) {
        if (!mbar_wait(r.act_bar, 0)) {
            record_status(a.status, RFP2_ETIMEOUT);
            *r.abort_flag = 1;
            return;
        }
        q = reinterpret_cast<const int8_t *>(act_q);
        d = reinterpret_cast<const float *>(act_d);
    }
    int c = 0;
    int64_t u = u0;
    while (u < u1) {
        const int g = (int)(u / tiles);
        const int t_begin = (int)(u % tiles);
        int64_t u_end = min(u1, (int64_t)(g + 1) * tiles);
        const int t_end = (int)(u_end - (int64_t)g * tiles);
        const int4 grp = a.ws.groups[g];
        bool ok = true;
        switch (grp.z) {
            case 1: ok = consume_group<1>(r, a, grp, t_begin, t_end, c, wg, a.WK > 1 ? wk : 0, lane, kb0, active, rowbytes, q, d, a.act_staged != 0); break;
            case 2: ok = consume_group<2>(r, a, grp, t_begin, t_end, c, wg, a.WK > 1 ? wk : 0, lane, kb0, active, rowbytes, q, d, a.act_staged != 0); break;
            case 3: ok = consume_group<3>(r, a, grp, t_begin, t_end, c, wg, a.WK > 1 ? wk : 0, lane, kb0, active, rowbytes, q, d, a.act_staged != 0); break;
            default: ok = consume_group<4>(r, a, grp, t_begin, t_end, c, wg, a.WK > 1 ? wk : 0, lane, kb0, active, rowbytes, q, d, a.act_staged != 0); break;
        }
        if (!ok) break;
        u = u_end;
    }
}

struct MoePlan {
    int WK, RG, nstages, tile_rows, grid, act_staged;
    size_t smem;
};

bool make_moe_plan(int64_t T, int64_t M, int64_t K, MoePlan &p) {
    const int KB = (int)(K / 32);
    int WK = (KB + 32 * kBpt - 1) / (32 * kBpt);
    int WKp = 1;
    while (WKp < WK) WKp *= 2;
    if (WKp > kConsumerWarps) return false;
    p.WK = WKp;
    p.RG = kConsumerWarps / WKp;
    p.tile_rows = p.RG * kChunksPerTile;
    const int chunk_bytes = p.RG * KB * 10;
    const int V = NextPow2<kGroupCols>::v;
    // stage every token's quantized activations in shared memory when they fit
    const size_t act = ((size_t)T * K + 15) / 16 * 16 + (size_t)T * KB * 4;
    p.act_staged = act <= 96 * 1024;
    const size_t act_smem = p.act_staged ? act : 0;
    int stages = 16;
    while (stages > 1 &&
           ring_bytes(stages, chunk_bytes, p.RG, p.WK, V) + act_smem > (size_t)kGemvSmemBudget)
        --stages;
    p.nstages = stages;
    p.smem = ring_bytes(stages, chunk_bytes, p.RG, p.WK, V) + act_smem;
    p.grid = sm_count(current_device());
    return p.smem <= 227 * 1024;
}

}  // namespace
}  // namespace rfp2

using namespace rfp2;

extern "C" size_t rfp2_moe_workspace_bytes(int64_t T, int64_t top_k, int64_t K) {
    if (T <= 0 || top_k <= 0 || K <= 0) return 0;
    return moe_ws_bytes(T, top_k, K);
}

extern "C" rfp2_status rfp2_moe_gemv(const uint8_t *W, int64_t E, int64_t M, int64_t K,
                                     const int32_t *ids, int64_t T, int64_t top_k, const float *x,
                                     float *y, void *workspace, size_t workspace_bytes,
                                     int32_t *dev_status, rfp2_stream_t stream) {
    if (!W || !ids || !x || !y) return RFP2_EINVAL;
    if (E <= 0 || M <= 0 || K <= 0 || T <= 0 || top_k <= 0) return RFP2_ESHAPE;
    if (T * top_k > kMaxPairs || M > (1 << 30) || K > (1 << 30) || E > 0x7FFFFFFF)
        return RFP2_ESHAPE;
    if (K % 256 != 0) return RFP2_EUNSUPPORTED;
    MoePlan p;
    if (!make_moe_plan(T, M, K, p)) return RFP2_EUNSUPPORTED;
    if (!workspace || workspace_bytes < moe_ws_bytes(T, top_k, K)) return RFP2_EWORKSPACE;
    if (!aligned(W, 16) || !aligned(x, 4) || !aligned(y, 4) || !aligned(ids, 4) ||
        !aligned(workspace, 256))
        return RFP2_EALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    MoeWs w = carve_ws(workspace, T, top_k, K);
    cudaError_t e = launch(moe_route_kernel, dim3(1), dim3(kRouteThreads), 0, s, true, ids,
                           (int)(T * top_k), E, (int)M, y, dev_status, w);
    if (e != cudaSuccess) return RFP2_ECUDA;
    e = launch_quantize(x, T, K, w.q, w.d, s, true);
    if (e != cudaSuccess) return RFP2_ECUDA;
    static std::mutex mu;
    static int configured[64] = {0};
    const int dev = current_device();
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && !configured[dev]) {
            if (set_smem_limit(moe_gemv_kernel, 227 * 1024) != cudaSuccess) return RFP2_ECUDA;
            configured[dev] = 1;
        }
    }
    MoeArgs a;
    a.W = W;
    a.expert_bytes = M * (K / 32) * 10;
    a.M = (int)M;
    a.K = (int)K;
    a.T = (int)T;
    a.top_k = (int)top_k;
    a.act_staged = p.act_staged;
    a.WK = p.WK;
    a.nstages = p.nstages;
    a.tile_rows = p.tile_rows;
    a.y = y;
    a.status = dev_status;
    a.ws = w;
    return from_cuda(launch(moe_gemv_kernel, dim3(p.grid), dim3(kGemvThreads), p.smem, s, true, a));
}
