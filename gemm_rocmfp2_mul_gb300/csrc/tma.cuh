// Tensor-map (TMA) helpers: host-side encoding of 2-D tiled tensor maps
// through the driver entry point (no link-time dependency on libcuda) and
// the device-side 2-D tile load into shared memory.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace rfp2 {

// Encode a 2-D tiled tensor map over a row-major matrix of `rows` x `cols`
// elements of `dtype` (row pitch `row_bytes`, a multiple of 16), with a box
// of box_cols x box_rows elements, no swizzle (or `swizzle`), out-of-bounds
// elements filled with zeros.  Returns false if the driver rejects it.
bool encode_tensor_map_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype,
                          uint64_t cols, uint64_t rows, uint64_t row_bytes, uint32_t box_cols,
                          uint32_t box_rows,
                          CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE);

// Encode a 3-D tiled tensor map: dims[0] contiguous elements, byte strides
// of dims 1 and 2 (multiples of 16), box `box` (box[0] * element size a
// multiple of 16), zero fill out of bounds.
bool encode_tensor_map_3d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype,
                          const uint64_t (&dims)[3], const uint64_t (&strides)[2],
                          const uint32_t (&box)[3],
                          CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE);

// 2-D tile load (box at element coordinates x = column, y = row) into shared
// memory, completing on `bar` (transaction bytes = full box, zero-filled out of
// bounds).  x * element size must be a multiple of 16 bytes.
RFP2_DEV void tma_load_2d(void *smem_dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// 2-D tile load into this CTA's shared memory whose completion is signalled
// on an mbarrier of either CTA of the pair (`bar_cluster`: shared::cluster
// address, e.g. the even CTA's barrier).
RFP2_DEV void tma_load_2d_pair(void *smem_dst, const CUtensorMap *map, int x, int y,
                               uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}

// 3-D tile load at element coordinates (x, y, z); x * element size must be a
// multiple of 16 bytes.
RFP2_DEV void tma_load_3d(void *smem_dst, const CUtensorMap *map, int x, int y, int z,
                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

// Same with an L2 cache-policy hint.
RFP2_DEV void tma_load_2d_hint(void *smem_dst, const CUtensorMap *map, int x, int y,
                               uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

RFP2_DEV void prefetch_tensor_map(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

}  // namespace rfp2
