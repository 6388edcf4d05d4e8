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

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// shared -> global tiled store of a box at (x, y), x >= 0 (the parts past the tensor's end are dropped)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, const void* src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(smem_u32(src))
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// the bulk stores this thread committed have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// ... and have completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Host: the driver's encoder, looked up once through the runtime (no link against libcuda).
bool encode_bf16_map_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t stride_bytes,
                        uint32_t box_inner, uint32_t box_rows);

// A bf16 tensor of `rank` (2 or 3) dimensions, innermost first (dims[0] contiguous), strides in bytes of
// dimensions 1.. (multiples of 16), a box of box[0..rank) elements written to shared memory in the
// 128-byte swizzle layout (box[0] * 2 <= 128 bytes; the destination 1024-byte aligned).
bool encode_bf16_map_sw128(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box);

}  // namespace ssm
