// Per-thread building blocks of the ROCmFP2 GEMV kernels (dense and MoE).
//
// Work split: a row of K/32 blocks is covered by WK warps; lane l of K-slice
// warp w owns the BPT consecutive blocks starting at (32*w + l) * BPT, keeps
// the matching int8 activations of all NC columns in registers (permuted into
// the lane order of expand_half) and walks down the rows of its row group.
// Every weight byte is expanded once and dotted with all NC columns (the
// multi-column reuse of "ROCmFP2 codebook research report", section
// "03 Runtime").  Per-row partial sums are combined across the warp with a
// transposing butterfly: V = R*NC partials per lane cost V-1+5-log2(V)
// shuffles in total instead of 5*V.
#pragma once

#include <stdint.h>

#include "common.cuh"
#include "rfp2_decode.cuh"

namespace rfp2 {

// Shared-memory budget of the streaming GEMV CTAs (one CTA per SM).
constexpr int kGemvSmemBudget = 200 * 1024;

template <int X>
struct NextPow2 {
    static constexpr int v = X <= 1 ? 1 : X <= 2 ? 2 : X <= 4 ? 4 : X <= 8 ? 8 : X <= 16 ? 16 : 32;
};
template <int X>
struct Log2 {
    static constexpr int v = X <= 1 ? 0 : 1 + Log2<X / 2>::v;
};
template <>
struct Log2<1> {
    static constexpr int v = 0;
};

// Largest blocks-per-thread for NC columns: keeps 8*BPT*NC activation words
// (<= 64 registers) resident.
#ifndef RFP2_GEMV_BPT12
#define RFP2_GEMV_BPT12 4
#endif
constexpr int bpt_max(int nc) { return nc <= 2 ? RFP2_GEMV_BPT12 : nc <= 4 ? 2 : 1; }

// Activations of one thread: [column][block][half][word] permuted int8 words
// and the per-block scale dA times 2^19 (see block_sum_2m19).
template <int NC, int BPT>
struct Act {
    uint32_t a[NC][BPT][2][4];
    float d[NC][BPT];
};

// Staged activations are stored with their 16-byte chunks XOR-swizzled inside
// every 128-byte group (chunk C lives at C ^ ((C >> 3) & 7)): a lane reads
// the 32 bytes of its block at a stride of 32*BPT bytes from its neighbour,
// which unswizzled puts every lane of a quarter warp on the same banks.
RFP2_DEV uint32_t act_swizzle(uint32_t chunk) { return chunk ^ ((chunk >> 3) & 7); }

// Load the thread's activations for columns cols[0..NC) (token rows of q/d).
// SWZ: q/d are the swizzled shared-memory copy made by load_act_to_smem
// (every warp of every CTA needs the same few KB, which from global memory
// piles all SMs onto the same L2 lines); otherwise plain global memory.
template <int NC, int BPT, bool SWZ>
RFP2_DEV void load_act(Act<NC, BPT> &A, const int8_t *q, const float *d, int K, int kb0,
                       bool active, const int (&cols)[NC]) {
    const int KB = K >> 5;
    const uint4 *q4 = reinterpret_cast<const uint4 *>(q);
#pragma unroll
    for (int n = 0; n < NC; ++n) {
#pragma unroll
        for (int b = 0; b < BPT; ++b) {
            if (active) {
                const uint32_t c0 = (uint32_t)(((int64_t)cols[n] * K + (int64_t)(kb0 + b) * 32) >> 4);
                const uint4 x0 = q4[SWZ ? act_swizzle(c0) : c0];
                const uint4 x1 = q4[SWZ ? act_swizzle(c0 + 1) : c0 + 1];
                permute_act_half(x0.x, x0.y, x0.z, x0.w, A.a[n][b][0]);
                permute_act_half(x1.x, x1.y, x1.z, x1.w, A.a[n][b][1]);
                A.d[n][b] = d[(int64_t)cols[n] * KB + kb0 + b] * 0x1p19f;
            } else {
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int i = 0; i < 4; ++i) A.a[n][b][h][i] = 0u;
                A.d[n][b] = 0.0f;
            }
        }
    }
}

// Load the thread's BPT blocks (10*BPT bytes at a 10*BPT-byte offset) from
// shared memory and dot them with all NC columns: out[n] += sum over blocks of
// dA * (d0 * S0 + d1 * S1).
template <int NC, int BPT>
RFP2_DEV void row_dot(const uint8_t *p, const Act<NC, BPT> &A, float (&out)[NC]) {
    constexpr int NW = BPT >= 2 ? 5 * BPT / 2 : 3;
    uint32_t v[NW];
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
#pragma unroll
    for (int b = 0; b < BPT; ++b) {
        Block k;
        if constexpr (BPT == 1) {
            k.lo = v[0];
            k.hi = v[1];
            k.scales = v[2];
        } else {
            k = block_from_words<BPT>(v, b);
        }
        uint32_t wlo[4], whi[4];
        expand_half(k.lo, wlo);
        expand_half(k.hi, whi);
        float s0, s1;
        placed_scale_pair(k.scales, s0, s1);
#pragma unroll
        for (int n = 0; n < NC; ++n)
            out[n] = fmaf(block_sum_2m19(wlo, whi, s0, s1, A.a[n][b][0], A.a[n][b][1]), A.d[n][b],
                          out[n]);
    }
}

// Transposing butterfly over the warp: on return, lane l holds the warp-wide
// sum of v[l >> (5 - log2 V)] (lanes are grouped in runs of 32/V).
template <int V>
RFP2_DEV float warp_transpose_reduce(float (&v)[V], int lane) {
    constexpr int L = Log2<V>::v;
#pragma unroll
    for (int s = 0; s < L; ++s) {
        const int half = V >> (s + 1);
        const int off = 16 >> s;
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    float t = v[0];
#pragma unroll
    for (int off = 16 >> L; off >= 1; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    return t;
}

}  // namespace rfp2

namespace rfp2 {

// Shared-memory ring and reduction state of a streaming GEMV CTA.
struct Ring {
    uint8_t *stages;        // [nstages][chunk_bytes]
    uint64_t *act_bar;      // activations staged in shared memory
    uint64_t *full;         // [nstages]   bulk copy landed
    uint64_t *empty;        // [nstages]   all consumer warps done with the stage
    uint64_t *redbar;       // [nstages][RG] K-slice partials written
    float *red;             // [nstages][RG][WK][V]
    volatile int *abort_flag;
    int nstages, chunk_bytes, RG, WK, V;
};

// Carve the ring out of dynamic shared memory.  Layout (ring_bytes): the
// stages, then 8-byte barriers (full, empty, reduction, activation) and the
// abort flag, then the reduction buffer; the total is a multiple of 128 so
// the caller can append 16-byte aligned regions (staged activations).
RFP2_DEV Ring carve_ring(uint8_t *smem, int nstages, int chunk_bytes, int RG, int WK, int V) {
    Ring r;
    r.stages = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)nstages * chunk_bytes);
    r.full = bars;
    r.empty = bars + nstages;
    r.redbar = bars + 2 * nstages;
    r.act_bar = bars + 2 * nstages + nstages * RG;
    r.abort_flag = reinterpret_cast<volatile int *>(r.act_bar + 1);
    r.red = reinterpret_cast<float *>(r.act_bar + 2);
    r.nstages = nstages;
    r.chunk_bytes = chunk_bytes;
    r.RG = RG;
    r.WK = WK;
    r.V = V;
    return r;
}

__host__ __device__ inline size_t ring_bytes(int nstages, int chunk_bytes, int RG, int WK, int V) {
    size_t s = (size_t)nstages * chunk_bytes;           // multiple of 16
    s += (size_t)(2 * nstages + nstages * RG + 2) * 8;  // barriers + abort flag
    s += (size_t)nstages * RG * WK * V * 4;             // reduction buffer
    return (s + 127) / 128 * 128;
}

// Initialise the ring's stage barriers (one thread, the producer) and make
// them visible to the async proxy; the caller may issue bulk copies on them
// right away, before the CTA-wide barrier.
RFP2_DEV void init_ring_stages(Ring &r, int consumer_warps, int act_arrivals = 32) {
    for (int s = 0; s < r.nstages; ++s) {
        mbar_init(&r.full[s], 1);
        mbar_init(&r.empty[s], consumer_warps);
    }
    mbar_init(r.act_bar, act_arrivals);
    *r.abort_flag = 0;
    fence_mbar_init();
}

// Initialise the reduction barriers (only used when a row spans several
// warps) with all threads of the CTA except `skip_warp`; call before the
// CTA-wide barrier.
RFP2_DEV void init_ring_reduction(Ring &r, int tid, int nthreads) {
    if (r.WK <= 1) return;
    for (int i = tid; i < r.nstages * r.RG; i += nthreads) mbar_init(&r.redbar[i], r.WK - 1);
}

// Producer side: issue chunk number c (rows*rowbytes bytes from src) into
// stage c % nstages, after the consumers released its previous use.
// Returns false on a timeout (status recorded, abort raised).
RFP2_DEV bool produce_chunk(Ring &r, int c, const uint8_t *src, uint32_t bytes, uint64_t policy,
                            int32_t *status) {
    const int s = c % r.nstages;
    if (c >= r.nstages) {
        if (!mbar_wait(&r.empty[s], ((c / r.nstages) - 1) & 1)) {
            record_status(status, RFP2_ETIMEOUT);
            *r.abort_flag = 1;
            return false;
        }
    }
    if (*r.abort_flag) return false;
    mbar_arrive_expect_tx(&r.full[s], bytes);
    bulk_g2s_stream(r.stages + (size_t)s * r.chunk_bytes, src, bytes, &r.full[s], policy);
    return true;
}

// Producer warp (all 32 lanes): copy the quantized activations (q: qbytes,
// d: dbytes, both multiples of 16, 16-byte aligned) into shared memory with
// ordinary loads, then arrive on the activation barrier (release: the stores
// are visible to the consumers that wait on it).  Ordinary loads do not queue
// behind the weight stream's bulk copies, so the activations land first.
RFP2_DEV void load_act_to_smem(Ring &r, int lane, uint8_t *dst_q, const int8_t *q,
                               uint32_t qbytes, uint8_t *dst_d, const float *d, uint32_t dbytes) {
    // all loads of a batch are issued before any store, so the copy costs one
    // memory round trip per 8 vectors per lane instead of one per vector
    const uint32_t nq = qbytes / 16, n = nq + dbytes / 16;
    const uint4 *sq = reinterpret_cast<const uint4 *>(q);
    const uint4 *sd = reinterpret_cast<const uint4 *>(d);
    uint4 *tq = reinterpret_cast<uint4 *>(dst_q);
    uint4 *td = reinterpret_cast<uint4 *>(dst_d);
    for (uint32_t base = 0; base < n; base += 8 * 32) {
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t i = base + j * 32 + lane;
            if (i < n) v[j] = i < nq ? sq[i] : sd[i - nq];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t i = base + j * 32 + lane;
            if (i < n) {
                if (i < nq) tq[act_swizzle(i)] = v[j];
                else td[i - nq] = v[j];
            }
        }
    }
    mbar_arrive(r.act_bar);
}

// Producer epilogue: the CTA must never retire with a copy into its shared
// memory in flight.  Without an abort every issued chunk is waited for by the
// consumers before they finish, so the producer leaves at once (waiting here
// was measured, in the dense GEMV, to keep a CTA resident up to ~0.8 us after
// its last consumer).  After an abort it waits (bounded) until the last use
// of every stage has landed.
RFP2_DEV void drain_ring(Ring &r, int issued, int32_t *status) {
    if (*r.abort_flag == 0) return;
    for (int c = max(0, issued - r.nstages); c < issued; ++c)
        if (!mbar_wait(&r.full[c % r.nstages], (c / r.nstages) & 1))
            record_status(status, RFP2_ETIMEOUT);
}

// Consumer side: one chunk.  Row group wg owns rows wg*R .. wg*R+R-1 of the
// chunk; rows[r] is the output row of the r-th and valid[r] says whether it
// exists.  The thread's BPT blocks sit at byte offset kb0*10 of each row.
// The R*NC partials are reduced over the warp with one transposing butterfly,
// then over the WK K-slice warps through the reduction buffer, and the
// K-slice-0 warp stores y for column n at ycol[n][row].  Returns false when
// the CTA must stop.
template <int NC, int BPT, int R>
RFP2_DEV bool consume_chunk(Ring &r, int c, int wg, int wk, int lane, int kb0, bool active,
                            int rowbytes, const int64_t (&rows)[R], const bool (&valid)[R],
                            const Act<NC, BPT> &A, float *const (&ycol)[NC], int32_t *status) {
    constexpr int V = NextPow2<R * NC>::v;
    constexpr int L = Log2<V>::v;
    const int s = c % r.nstages;
    const uint32_t par = (c / r.nstages) & 1;
    if (*r.abort_flag) return false;
    if (!mbar_wait(&r.full[s], par)) {
        record_status(status, RFP2_ETIMEOUT);
        *r.abort_flag = 1;
        return false;
    }
    float vals[V];
#pragma unroll
    for (int i = 0; i < V; ++i) vals[i] = 0.0f;
    // Straight-line over the R rows so their decodes interleave: a row past
    // the end of the slab still lies inside the stage and is computed but
    // never stored; an inactive lane (beyond K) reads the row start and has
    // zero activations.
    const uint8_t *base = r.stages + (size_t)s * r.chunk_bytes + (size_t)wg * R * rowbytes +
                          (active ? kb0 * 10 : 0);
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        float o[NC];
#pragma unroll
        for (int n = 0; n < NC; ++n) o[n] = 0.0f;
        row_dot<NC, BPT>(base + rr * rowbytes, A, o);
#pragma unroll
        for (int n = 0; n < NC; ++n) vals[rr * NC + n] = o[n];
    }
    float total = warp_transpose_reduce<V>(vals, lane);
    const int idx = lane >> (5 - L);
    const bool writer = (lane & ((32 >> L) - 1)) == 0;
    bool ok = true;
    if (r.WK > 1) {
        float *slot = r.red + (size_t)(s * r.RG + wg) * r.WK * V;
        if (wk != 0) {
            if (writer) slot[wk * V + idx] = total;
            __syncwarp();
            if (lane == 0) mbar_arrive(&r.redbar[s * r.RG + wg]);
        } else {
            if (!mbar_wait(&r.redbar[s * r.RG + wg], par)) {
                record_status(status, RFP2_ETIMEOUT);
                *r.abort_flag = 1;
                ok = false;
            } else if (writer) {
                for (int j = 1; j < r.WK; ++j) total += slot[j * V + idx];
            }
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&r.empty[s]);
    if (!ok) return false;
    if (wk == 0 && writer && idx < R * NC) {
#pragma unroll
        for (int rr = 0; rr < R; ++rr)
#pragma unroll
            for (int n = 0; n < NC; ++n)
                if (idx == rr * NC + n && valid[rr]) ycol[n][rows[rr]] = total;
    }
    return true;
}

}  // namespace rfp2
