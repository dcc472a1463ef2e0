// Shared device and host helpers of librfp2 (sm_103a).
//
// Device side: inline-PTX wrappers for mbarriers, 1-D bulk async copies
// (global -> shared, completing on an mbarrier), programmatic dependent launch
// and a bounded wait that gives up after a fixed time and reports
// RFP2_ETIMEOUT instead of spinning forever.
//
// Host side: argument-check helpers, per-device SM counts and a launcher that
// optionally sets the programmatic-stream-serialization attribute.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "rfp2.h"

#define RFP2_DEV __device__ __forceinline__

namespace rfp2 {

// ---------------------------------------------------------------------------
// Device helpers

RFP2_DEV uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

RFP2_DEV uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

RFP2_DEV void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

RFP2_DEV void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

RFP2_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

RFP2_DEV void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One try_wait: returns once the phase with `parity` has completed or after a
// short, hardware-defined interval.
RFP2_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Time limit of every device wait.  Far above any legitimate wait (the
// longest kernel here runs for about a millisecond) and short enough that a
// broken pipeline returns an error instead of holding the GPU.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Waits for the phase with `parity` of `bar` to complete.  Returns false if
// the time limit ran out (the caller records RFP2_ETIMEOUT and winds down).
RFP2_DEV bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// The same for a wait that may last long (a producer waiting for its
// consumers, possibly for the whole of the previous kernel): it sleeps between
// probes so that it does not take issue slots from the warps doing the work.
RFP2_DEV bool mbar_wait_sleepy(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        __nanosleep(256);
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// ---- clusters ----------------------------------------------------------------
RFP2_DEV uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Shared::cluster address of the variable at `p`'s offset in CTA `rank` of
// this cluster.
RFP2_DEV uint32_t cluster_map(const void *p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(p)), "r"(rank));
    return a;
}
// Arrive on an mbarrier given by its shared::cluster address (any CTA of the
// cluster).
RFP2_DEV void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
// Orders this thread's earlier generic-proxy writes to shared memory before
// later async-proxy reads of it (tensor-core operands, bulk copies).
RFP2_DEV void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// The same with the default (CTA-scope release) semantics, for a producer
// whose data is handed over by a proxy fence and an mbarrier phase (the
// cluster-scope release costs about a microsecond per arrival).
RFP2_DEV void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// All threads of all CTAs of the cluster.
RFP2_DEV void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// 1-D bulk async copy global -> shared; completion is signalled on `bar`
// (transaction bytes).  Both addresses 16-byte aligned, bytes % 16 == 0.
RFP2_DEV void bulk_g2s(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Same, with an L2 evict-first hint: weights are streamed once per call.
RFP2_DEV void bulk_g2s_stream(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar,
                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
        "[%1], %2, [%3], %4;" ::"r"(smem_addr(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Prefetch `bytes` (a multiple of 16, 16-byte aligned address) of global
// memory into L2.  L2 is the point of coherence, so a prefetch can never make
// a later read return stale data.
RFP2_DEV void bulk_prefetch_l2(const void *gsrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gsrc), "r"(bytes) : "memory");
}

RFP2_DEV uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Programmatic dependent launch: wait for the preceding grid's memory, and
// allow the next grid in the stream to begin launching.
RFP2_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
RFP2_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

RFP2_DEV void record_status(int32_t *dev_status, int32_t code) {
    if (dev_status) atomicCAS(reinterpret_cast<int *>(dev_status), 0, code);
}

// Named barrier over `nthreads` threads (a multiple of 32).
RFP2_DEV void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// Host helpers

int sm_count(int device);
int current_device();
// rfp2_set_weight_prefetch: may a kernel read weights before the work
// enqueued ahead of it on the stream has completed?
bool weight_prefetch();
cudaError_t launch_status();  // cudaGetLastError wrapper

inline bool aligned(const void *p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

inline rfp2_status from_cuda(cudaError_t e) { return e == cudaSuccess ? RFP2_OK : RFP2_ECUDA; }

// Launch `kernel` with an optional programmatic-stream-serialization
// attribute (the kernel may start while the previous kernel in the stream is
// still running; it must call pdl_wait() before touching that kernel's
// outputs).
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                   cudaStream_t stream, bool pdl, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Sets the dynamic shared memory limit of `kernel` once per device.
template <typename K>
cudaError_t set_smem_limit(K kernel, int bytes) {
    return cudaFuncSetAttribute(reinterpret_cast<const void *>(kernel),
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace rfp2
