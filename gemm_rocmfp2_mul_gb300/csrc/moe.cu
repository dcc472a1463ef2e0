// MoE bulk-expert GEMV: y[t, j, :] = W[ids[t, j]] x_t for T tokens routed to
// top_k of E ROCmFP2 experts (MUL_MAT_ID run as a GEMV over the routed
// experts' rows for a few tokens: "HRX on the Radeon iGPU", section "MoE
// decode and the kernel cache"; expand-once multi-column reuse: "ROCmFP2
// codebook research report", section "03 Runtime").
//
// Three launches chained with programmatic dependent launch:
//  1. route (one CTA): validates the ids (an id outside [0, E) is never
//     dereferenced: its output row is filled with NaN and RFP2_EBADID is
//     recorded), ranks the (token, slot) pairs by expert (several threads per
//     pair) and cuts each expert's run into groups of at most two pairs
//     (two tokens' activations fit in registers beside four rows per warp).
//     Groups go to the workspace.
//  2. quantize the T tokens once (Q8_1-style blocks) into the workspace.
//  3. moe_gemv (persistent, one CTA per SM): work units are (group, tile of
//     rows of that expert); CTA i takes a contiguous range of units, its
//     producer warp streams the expert rows into the shared-memory ring and
//     the consumer warps expand every block once for the group's tokens.
//     The group list, the pair order and the quantized tokens are first
//     copied into shared memory by all threads together (one memory round
//     trip).  Expert offsets are 64-bit.
#include <mutex>

#include <algorithm>

#include "common.cuh"
#include "gemv_core.cuh"
#include "quantize.cuh"

namespace rfp2 {
namespace {

#ifndef RFP2_MOE_WARPS
#define RFP2_MOE_WARPS 16
#endif
#ifndef RFP2_MOE_COLS
#define RFP2_MOE_COLS 2
#endif
#ifndef RFP2_MOE_ROWS
#define RFP2_MOE_ROWS 4
#endif
#ifndef RFP2_MOE_CHUNKS_PER_TILE
#define RFP2_MOE_CHUNKS_PER_TILE 1
#endif
constexpr int kConsumerWarps = RFP2_MOE_WARPS;
constexpr int kGemvThreads = (kConsumerWarps + 1) * 32;
constexpr int kGroupCols = RFP2_MOE_COLS;  // tokens per group (activation registers)
constexpr int kBpt = 2;                    // blocks per thread
constexpr int kRows = RFP2_MOE_ROWS;       // rows per warp per chunk
constexpr int kChunksPerTile = RFP2_MOE_CHUNKS_PER_TILE;  // rows per unit = chunks of RG*kRows
// Chunks whose partials a consumer warp keeps in registers before one warp
// reduction covers them (at most 16 values: kRows x tokens per chunk).
template <int NC>
constexpr int defer_chunks() {
    return kRows * NC <= 4 ? 4 : kRows * NC <= 8 ? 2 : 1;
}
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

// Shared memory of the routing pass: sid, gidx and erank (ints), left
// (shorts) and flag (bytes), P entries each.
size_t route_smem_bytes(int P) { return (size_t)P * (4 + 4 + 4 + 2 + 1) + 16; }

RFP2_DEV void moe_route_body(const int32_t *__restrict__ ids, int P, int64_t E, int M, float *y,
                            int32_t *status, const MoeWs &w, int *rsm) {
    int *sid = rsm;              // expert of pair p, -1 if invalid
    int *gidx = sid + P;         // by sorted position: group-start flag, then group index
    int *erank = gidx + P;       // by sorted position: expert
    short *left = reinterpret_cast<short *>(erank + P);  // pairs left in the expert run
    unsigned char *flag = reinterpret_cast<unsigned char *>(left + P);
    __shared__ int warp_sums[32];
    const int tid = threadIdx.x;
    int nvalid = 0;
    for (int base = 0; base < P; base += blockDim.x) {
        const int p = base + tid;
        bool ok = false;
        if (p < P) {
            const int32_t e = ids[p];
            ok = e >= 0 && (int64_t)e < E;
            sid[p] = ok ? e : -1;
            if (!ok) record_status(status, RFP2_EBADID);
        }
        nvalid += __syncthreads_count(ok);
    }
    // NaN rows for invalid pairs (their ids are never used as expert offsets)
    if (nvalid < P) {
        for (int64_t i = tid; i < (int64_t)P * M; i += blockDim.x)
            if (sid[i / M] < 0) y[i] = __int_as_float(0x7fc00000);
    }
    // Rank of each valid pair by (expert, p), its position inside the expert's
    // run and the run length: tpp threads per pair each scan every tpp-th pair,
    // then sum over their aligned lane group.
    int tpp = 1;
    while (tpp < 32 && tpp * P < (int)blockDim.x) tpp *= 2;
    const int ppr = blockDim.x / tpp, j = tid & (tpp - 1);
    for (int p0 = 0; p0 < P; p0 += ppr) {
        const int p = p0 + tid / tpp;
        const int e = p < P ? sid[p] : -1;
        int rank = 0, before = 0, count = 0;
        if (e >= 0) {
            for (int p2 = j; p2 < P; p2 += tpp) {
                const int e2 = sid[p2];
                if (e2 < 0) continue;
                rank += (e2 < e) || (e2 == e && p2 < p);
                before += e2 < e;
                count += e2 == e;
            }
        }
        for (int off = 1; off < tpp; off <<= 1) {
            rank += __shfl_xor_sync(0xffffffffu, rank, off);
            before += __shfl_xor_sync(0xffffffffu, before, off);
            count += __shfl_xor_sync(0xffffffffu, count, off);
        }
        if (e >= 0 && j == 0) {
            const int pos = rank - before;
            w.sorted[rank] = p;
            erank[rank] = e;
            flag[rank] = (pos % kGroupCols) == 0;
            gidx[rank] = (pos % kGroupCols) == 0;
            left[rank] = (short)(count - pos);
        }
    }
    __syncthreads();
    block_exclusive_scan(gidx, nvalid, warp_sums);  // gidx[r] = starts before r
    for (int r = tid; r < nvalid; r += blockDim.x) {
        if (!flag[r]) continue;
        w.groups[gidx[r]] = make_int4(erank[r], r, min(kGroupCols, (int)left[r]), 0);
    }
    if (tid == 0) {
        w.header[0] = nvalid > 0 ? gidx[nvalid - 1] + flag[nvalid - 1] : 0;
        w.header[1] = nvalid;
    }
}

// One launch for both inputs of the MoE GEMV: CTA 0 routes (the pass above),
// the other CTAs quantize the tokens, one warp per 32-value block.
__global__ void __launch_bounds__(kRouteThreads, 1)
    moe_prep_kernel(const int32_t *__restrict__ ids, int P, int64_t E, int M, float *y,
                    int32_t *status, MoeWs w, const float *__restrict__ x, int64_t nblocks) {
    extern __shared__ __align__(16) int rsm[];
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0) {
        moe_route_body(ids, P, E, M, y, status, w, rsm);
        return;
    }
    const int warps = blockDim.x >> 5;
    for (int64_t b = (int64_t)(blockIdx.x - 1) * warps + (threadIdx.x >> 5); b < nblocks;
         b += (int64_t)(gridDim.x - 1) * warps)
        quantize_block_warp(x, b, threadIdx.x & 31, w.q, w.d);
}

struct MoeArgs {
    const uint8_t *W;
    int64_t expert_bytes;
    int M, K, T, top_k, WK, nstages, tile_rows;
    int act_staged;   // token activations staged in shared memory
    int meta_staged;  // group list and pair order staged in shared memory
    float *y;
    int32_t *status;
    MoeWs ws;
};

// Consumer side, one warp per row (no K-slices): decode chunk c into the R x
// NC lane partials `part` and release its stage at once; the reduction over
// the warp is left to the caller.  Returns false when the CTA must stop.
template <int NC, int BPT, int R>
RFP2_DEV bool decode_chunk(Ring &r, int c, int wg, int lane, int kb0, bool active, int rowbytes,
                           const Act<NC, BPT> &A, float (&part)[R][NC], int32_t *status) {
    const int s = c % r.nstages;
    if (!mbar_try_wait(&r.full[s], (c / r.nstages) & 1)) {
        if (*r.abort_flag || !mbar_wait(&r.full[s], (c / r.nstages) & 1)) {
            record_status(status, RFP2_ETIMEOUT);
            *r.abort_flag = 1;
            return false;
        }
    }
    const uint8_t *base = r.stages + (size_t)s * r.chunk_bytes + (size_t)wg * R * rowbytes +
                          (active ? kb0 * 10 : 0);
#pragma unroll
    for (int rr = 0; rr < R; ++rr) row_dot<NC, BPT>(base + rr * rowbytes, A, part[rr]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&r.empty[s]);
    return true;
}

template <int NC>
__device__ bool consume_group(Ring &r, const MoeArgs &a, int4 grp, int t_begin, int t_end, int &c,
                              int wg, int wk, int lane, int kb0, bool active, int rowbytes,
                              const int8_t *q, const float *d, bool staged, const int *sorted) {
    int cols[NC];
    float *ycol[NC];
#pragma unroll
    for (int n = 0; n < NC; ++n) {
        const int pair = sorted[grp.y + n];
        cols[n] = pair / a.top_k;
        ycol[n] = a.y + (int64_t)pair * a.M;
    }
    Act<NC, kBpt> A;
    if (staged)
        load_act<NC, kBpt, true>(A, q, d, a.K, kb0, active, cols);
    else
        load_act<NC, kBpt, false>(A, q, d, a.K, kb0, active, cols);
    const int cr = r.RG * kRows;
    constexpr int VS = kRows * NC;
    constexpr int D = defer_chunks<NC>();
    if (D > 1 && a.WK == 1) {
        // A warp owns whole rows: the partials of D consecutive chunks stay
        // in registers (each chunk's stage is released as soon as it is
        // decoded) and one transposing reduction covers them, so the warps
        // do not all stall on a shuffle chain after every chunk.
        constexpr int VD = NextPow2<D * VS>::v;
        constexpr int LD = Log2<VD>::v;
        const int idx = lane >> (5 - LD);
        const bool writer = (lane & ((32 >> LD) - 1)) == 0 && idx < D * VS;
        const int vj = idx / VS, vr = (idx / NC) % kRows, vn = idx % NC;
        float *yw = ycol[0];
#pragma unroll
        for (int n = 1; n < NC; ++n)
            if (vn == n) yw = ycol[n];
        int t = t_begin, ch = 0;
        while (t < t_end) {
            float part[D][kRows][NC];
#pragma unroll
            for (int j = 0; j < D; ++j)
#pragma unroll
                for (int rr = 0; rr < kRows; ++rr)
#pragma unroll
                    for (int n = 0; n < NC; ++n) part[j][rr][n] = 0.0f;
            int wrow = 0, wlim = 0;  // the writer's row and its tile's end
#pragma unroll
            for (int j = 0; j < D; ++j) {
                if (t < t_end) {
                    const int r0 = t * a.tile_rows;
                    const int r1 = min(a.M, r0 + a.tile_rows);
                    if (j == vj) {
                        wrow = r0 + ch * cr + wg * kRows + vr;
                        wlim = r1;
                    }
                    if (!decode_chunk<NC, kBpt, kRows>(r, c, wg, lane, kb0, active, rowbytes, A,
                                                       part[j], a.status))
                        return false;
                    ++c;
                    if (++ch == (r1 - r0 + cr - 1) / cr) {
                        ch = 0;
                        ++t;
                    }
                }
            }
            float vals[VD];
#pragma unroll
            for (int i = 0; i < VD; ++i)
                vals[i] = i < D * VS ? part[i / VS][(i / NC) % kRows][i % NC] : 0.0f;
            const float total = warp_transpose_reduce<VD>(vals, lane);
            if (writer && wrow < wlim) yw[wrow] = total;
        }
        return true;
    }
    for (int t = t_begin; t < t_end; ++t) {
        const int r0 = t * a.tile_rows;
        const int r1 = min(a.M, r0 + a.tile_rows);
        const int nch = (r1 - r0 + cr - 1) / cr;
        for (int ch = 0; ch < nch; ++ch, ++c) {
            int64_t rows[kRows];
            bool valid[kRows];
#pragma unroll
            for (int rr = 0; rr < kRows; ++rr) {
                rows[rr] = r0 + (int64_t)ch * cr + wg * kRows + rr;
                valid[rr] = rows[rr] < r1;
            }
            if (!consume_chunk<NC, kBpt, kRows>(r, c, wg, wk, lane, kb0, active, rowbytes, rows,
                                                valid, A, ycol, a.status))
                return false;
        }
    }
    return true;
}

// Cooperative copy, global -> shared, of the token activations (q swizzled,
// then d) and of the group list and pair order: every thread keeps up to
// eight 16-byte loads in flight, so the whole copy costs about one memory
// round trip.
__device__ void stage_inputs(const MoeArgs &a, int ngroups, int nvalid, uint8_t *act_q,
                             uint8_t *act_d, int4 *sgroups, int *ssorted) {
    const uint32_t nq = a.act_staged ? (uint32_t)a.T * a.K / 16 : 0;
    const uint32_t nd = a.act_staged ? (uint32_t)a.T * (a.K / 32) * 4 / 16 : 0;
    const uint32_t ng = a.meta_staged ? (uint32_t)ngroups : 0;
    const uint32_t ns = a.meta_staged ? (uint32_t)(nvalid + 3) / 4 : 0;
    const uint32_t n = nq + nd + ng + ns;
    const uint4 *srcq = reinterpret_cast<const uint4 *>(a.ws.q);
    const uint4 *srcd = reinterpret_cast<const uint4 *>(a.ws.d);
    const uint4 *srcg = reinterpret_cast<const uint4 *>(a.ws.groups);
    const uint4 *srcs = reinterpret_cast<const uint4 *>(a.ws.sorted);
    uint4 *dq = reinterpret_cast<uint4 *>(act_q);
    uint4 *dd = reinterpret_cast<uint4 *>(act_d);
    uint4 *dg = reinterpret_cast<uint4 *>(sgroups);
    uint4 *ds = reinterpret_cast<uint4 *>(ssorted);
    for (uint32_t base = 0; base < n; base += 8 * blockDim.x) {
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t i = base + j * blockDim.x + threadIdx.x;
            if (i >= n) continue;
            if (i < nq) { v[j] = srcq[i]; continue; }
            i -= nq;
            if (i < nd) { v[j] = srcd[i]; continue; }
            i -= nd;
            if (i < ng) { v[j] = srcg[i]; continue; }
            v[j] = srcs[i - ng];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t i = base + j * blockDim.x + threadIdx.x;
            if (i >= n) continue;
            if (i < nq) { dq[act_swizzle(i)] = v[j]; continue; }
            i -= nq;
            if (i < nd) { dd[i] = v[j]; continue; }
            i -= nd;
            if (i < ng) { dg[i] = v[j]; continue; }
            ds[i - ng] = v[j];
        }
    }
}

__global__ void __launch_bounds__(kGemvThreads, 1) moe_gemv_kernel(MoeArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int KB = a.K >> 5;
    const int rowbytes = KB * 10;
    const int RG = kConsumerWarps / a.WK;
    Ring r = carve_ring(smem, a.nstages, RG * kRows * rowbytes, RG, a.WK,
                        NextPow2<kRows * kGroupCols>::v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t qbytes = a.act_staged ? (uint32_t)a.T * a.K : 0;
    const uint32_t dbytes = a.act_staged ? (uint32_t)a.T * KB * 4 : 0;
    uint8_t *act_q = smem + ring_bytes(a.nstages, RG * kRows * rowbytes, RG, a.WK,
                                       NextPow2<kRows * kGroupCols>::v);
    uint8_t *act_d = act_q + ((qbytes + 15) & ~15u);
    int4 *sgroups = reinterpret_cast<int4 *>(act_d + ((dbytes + 15) & ~15u));
    int *ssorted = reinterpret_cast<int *>(sgroups + (a.meta_staged ? a.T * a.top_k : 0));
    if (threadIdx.x == kConsumerWarps * 32) init_ring_stages(r, kConsumerWarps);
    init_ring_reduction(r, threadIdx.x, kConsumerWarps * 32);
    // the group list and the quantized tokens come from the two launches before
    pdl_wait();
    pdl_launch_dependents();
    const int ngroups = a.ws.header[0];
    const int nvalid = a.ws.header[1];
    stage_inputs(a, ngroups, nvalid, act_q, act_d, sgroups, ssorted);
    __syncthreads();
    const int4 *groups = a.meta_staged ? sgroups : a.ws.groups;
    const int *sorted = a.meta_staged ? ssorted : a.ws.sorted;
    const int tiles = (a.M + a.tile_rows - 1) / a.tile_rows;
    // units (group, row tile) split into contiguous, balanced CTA ranges
    const int units = ngroups * tiles;
    const int per = units / (int)gridDim.x, extra = units % (int)gridDim.x;
    const int bx = blockIdx.x;
    const int u0 = bx * per + min(bx, extra);
    const int u1 = u0 + per + (bx < extra ? 1 : 0);

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int c = 0;
            bool ok = true;
            for (int u = u0; u < u1 && ok; ++u) {
                const int g = u / tiles, t = u - g * tiles;
                const int4 grp = groups[g];
                const uint8_t *base = a.W + (int64_t)grp.x * a.expert_bytes;
                const int r0 = t * a.tile_rows;
                const int r1 = min(a.M, r0 + a.tile_rows);
                for (int row = r0; row < r1 && ok; row += RG * kRows, ++c) {
                    const int rows = min(RG * kRows, r1 - row);
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
    const int8_t *q = a.act_staged ? reinterpret_cast<const int8_t *>(act_q) : a.ws.q;
    const float *d = a.act_staged ? reinterpret_cast<const float *>(act_d) : a.ws.d;
    int c = 0;
    int u = u0;
    while (u < u1) {
        const int g = u / tiles;
        const int t_begin = u - g * tiles;
        const int u_end = min(u1, (g + 1) * tiles);
        const int t_end = u_end - g * tiles;
        const int4 grp = groups[g];
        bool ok = true;
        const int wkk = a.WK > 1 ? wk : 0;
        if (kGroupCols >= 2 && grp.z >= 2) {
            if constexpr (kGroupCols >= 4) {
                if (grp.z == 4)
                    ok = consume_group<4>(r, a, grp, t_begin, t_end, c, wg, wkk, lane, kb0, active,
                                          rowbytes, q, d, a.act_staged != 0, sorted);
                else if (grp.z == 3)
                    ok = consume_group<3>(r, a, grp, t_begin, t_end, c, wg, wkk, lane, kb0, active,
                                          rowbytes, q, d, a.act_staged != 0, sorted);
                else
                    ok = consume_group<2>(r, a, grp, t_begin, t_end, c, wg, wkk, lane, kb0, active,
                                          rowbytes, q, d, a.act_staged != 0, sorted);
            } else {
                ok = consume_group<2>(r, a, grp, t_begin, t_end, c, wg, wkk, lane, kb0, active,
                                      rowbytes, q, d, a.act_staged != 0, sorted);
            }
        } else {
            ok = consume_group<1>(r, a, grp, t_begin, t_end, c, wg, wkk, lane, kb0, active,
                                  rowbytes, q, d, a.act_staged != 0, sorted);
        }
        if (!ok) break;
        u = u_end;
    }
}

struct MoePlan {
    int WK, RG, nstages, tile_rows, grid, act_staged, meta_staged;
    size_t smem;
};

bool make_moe_plan(int64_t T, int64_t top_k, int64_t M, int64_t K, MoePlan &p) {
    const int KB = (int)(K / 32);
    int WK = (KB + 32 * kBpt - 1) / (32 * kBpt);
    int WKp = 1;
    while (WKp < WK) WKp *= 2;
    if (WKp > kConsumerWarps) return false;
    p.WK = WKp;
    p.RG = kConsumerWarps / WKp;
    p.tile_rows = p.RG * kRows * kChunksPerTile;
    const int chunk_bytes = p.RG * kRows * KB * 10;
    const int V = NextPow2<kRows * kGroupCols>::v;
    // stage every token's quantized activations in shared memory when they fit
    const size_t act = ((size_t)T * K + 15) / 16 * 16 + (size_t)T * KB * 4;
    p.act_staged = act <= 96 * 1024;
    // the group list (<= T*top_k int4) and the pair order (T*top_k ints)
    const size_t meta = (size_t)T * top_k * 16 + ((size_t)T * top_k * 4 + 15) / 16 * 16;
    p.meta_staged = meta <= 16 * 1024;
    const size_t act_smem = (p.act_staged ? act : 0) + (p.meta_staged ? meta : 0);
    int stages = 32;
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
    if (!make_moe_plan(T, top_k, M, K, p)) return RFP2_EUNSUPPORTED;
    if (!workspace || workspace_bytes < moe_ws_bytes(T, top_k, K)) return RFP2_EWORKSPACE;
    if (!aligned(W, 16) || !aligned(x, 4) || !aligned(y, 4) || !aligned(ids, 4) ||
        !aligned(workspace, 256))
        return RFP2_EALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    MoeWs w = carve_ws(workspace, T, top_k, K);
    static std::mutex mu;
    static int configured[64] = {0};
    const int dev = current_device();
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && !configured[dev]) {
            if (set_smem_limit(moe_gemv_kernel, 227 * 1024) != cudaSuccess ||
                set_smem_limit(moe_prep_kernel, (int)route_smem_bytes(kMaxPairs)) != cudaSuccess)
                return RFP2_ECUDA;
            configured[dev] = 1;
        }
    }
    const int64_t nblocks = T * (K / 32);
    const int64_t qctas = std::min<int64_t>((nblocks + kRouteThreads / 32 - 1) / (kRouteThreads / 32),
                                            4 * (int64_t)sm_count(dev));
    cudaError_t e = launch(moe_prep_kernel, dim3((unsigned)(1 + qctas)), dim3(kRouteThreads),
                           route_smem_bytes((int)(T * top_k)), s, true, ids, (int)(T * top_k), E,
                           (int)M, y, dev_status, w, x, nblocks);
    if (e != cudaSuccess) return RFP2_ECUDA;
    MoeArgs a;
    a.W = W;
    a.expert_bytes = M * (K / 32) * 10;
    a.M = (int)M;
    a.K = (int)K;
    a.T = (int)T;
    a.top_k = (int)top_k;
    a.act_staged = p.act_staged;
    a.meta_staged = p.meta_staged;
    a.WK = p.WK;
    a.nstages = p.nstages;
    a.tile_rows = p.tile_rows;
    a.y = y;
    a.status = dev_status;
    a.ws = w;
    return from_cuda(launch(moe_gemv_kernel, dim3(p.grid), dim3(kGemvThreads), p.smem, s, true, a));
}
