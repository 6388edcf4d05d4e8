// 2-D tiled bulk-tensor copies (TMA) into shared memory, completing on an mbarrier, and the host side
// that encodes their tensor maps.  A map describes a row-major bf16 matrix (inner dimension `inner`
// elements, `rows` rows, row stride `stride_bytes`) and the box one copy moves; a copy at coordinates
// (x, y) fills the box from element x of row y, with zeros where the box leaves the matrix (x may be
// negative).  Requirements, checked by the caller before choosing this path: 16-byte-aligned base and
// row stride, box inner size a multiple of 16 bytes, and every x times 2 bytes a multiple of 16.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "bulk_copy.cuh"

namespace ssm {

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Host: the driver's encoder, looked up once through the runtime (no link against libcuda).
bool encode_bf16_map_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t stride_bytes,
                        uint32_t box_inner, uint32_t box_rows);

}  // namespace ssm
