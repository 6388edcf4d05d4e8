// Fifth-generation tensor cores (tcgen05) for sm_100-family GPUs, as inline PTX: tensor-memory (TMEM)
// allocation, single-thread MMA issue with bf16 operands from shared memory and an fp32 accumulator in
// TMEM, completion through an mbarrier, and the per-warp TMEM loads of an epilogue.
//
// Operand tiles are in the 128-byte swizzle layout that a TMA copy with SWIZZLE_128B writes.  K-major:
// rows of 64 bf16 (128 bytes), 8-row atoms of 1024 bytes in which the 16-byte chunk c of row r sits at
// chunk c ^ (r % 8); a tile with K > 64 is a sequence of such 64-wide K blocks, each (rows x 128) bytes.
// Tiles start on 1024-byte boundaries.  One MMA consumes K = 16 (32 bytes of every row); the k-th step
// of a block starts 32 k bytes into it, and the hardware applies the swizzle to the computed addresses.
//
// TMEM: 128 lanes x 512 columns of 32 bits per SM.  An M = 128 accumulator puts row i in lane i and
// column j in column (base + j).  Warp w of a warpgroup may only touch lanes 32 (w % 4) .. 32 (w % 4) + 31.
#pragma once

#include <cstdint>

#include "bulk_copy.cuh"

namespace ssm {
namespace tc {

// one full warp: allocate `ncols` TMEM columns (a power of two, 32..512); the base address lands in *dst
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// one full warp (the one that allocated)
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols) : "memory");
}

// order tcgen05 work across a thread barrier: "before" ahead of the barrier, "after" behind it
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// shared-memory writes of this thread become visible to the async proxy (MMA operand reads, TMA)
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled operand starting at `addr` (a shared
// address; the tile's 1024-byte atoms must be aligned): stride between 8-row groups 1024 bytes, the
// leading offset unused by this layout, descriptor version 1, swizzle mode 2 (128 bytes).
__device__ __forceinline__ uint64_t desc_k_sw128(uint32_t addr) {
    uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Shared-memory matrix descriptor of an MN-major, 128-byte-swizzled operand: lines of 64 M (or N)
// elements (128 bytes), one per K index, 8-line atoms of 1024 bytes; `mn_stride` bytes between the
// 64-element blocks along M (N), `k_stride` bytes between 8-line groups along K.
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t addr, uint32_t mn_stride, uint32_t k_stride) {
    uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((mn_stride >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((k_stride >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 D, shape M x N; B K-major, A K-major or
// (a_mn) MN-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn = false) {
    return (1u << 4)                                   // D format: f32
           | (1u << 7)                                 // A format: bf16
           | (1u << 10)                                // B format: bf16
           | (a_mn ? (1u << 15) : 0u)                  // A major-ness: MN
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// D[tmem] = A B^T (accumulate = 0) or D += A B^T; A is M x 16, B is N x 16, both K-major.  One thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same product with A (M x 16, K-major) in tensor memory at `a_tmem`: row i in lane i, two consecutive
// K elements per 32-bit column (the lower one in the low half).  One thread.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 8 consecutive 32-bit columns of this thread's lane from `taddr` (lane in bits 31..16); the whole warp
// stores, each thread its own lane.  tmem_wait_st waits for the warp's stores.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// one arrival on `bar` once every MMA this thread issued before has completed
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 consecutive 32-bit columns of this thread's lane, starting at `taddr` (lane in bits 31..16), waited
// for inside the same statement so that no use of the registers can be scheduled ahead of the load
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive 32-bit columns of this thread's lane (as tmem_ld32)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// n blocks of 16 consecutive columns of this thread's lane, at taddr[0..n), all waited for at once
template <int kBlocks>
__device__ __forceinline__ void tmem_ld16xn(const uint32_t (&taddr)[kBlocks], float (&v)[kBlocks][16]) {
    static_assert(kBlocks == 2 || kBlocks == 4, "blocks");
    uint32_t r[kBlocks][16];
#define SSM_TC_LD16(i)                                                                                          \
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, " \
                 "%13, %14, %15}, [%16];"                                                                       \
                 : "=r"(r[i][0]), "=r"(r[i][1]), "=r"(r[i][2]), "=r"(r[i][3]), "=r"(r[i][4]), "=r"(r[i][5]),      \
                   "=r"(r[i][6]), "=r"(r[i][7]), "=r"(r[i][8]), "=r"(r[i][9]), "=r"(r[i][10]), "=r"(r[i][11]),   \
                   "=r"(r[i][12]), "=r"(r[i][13]), "=r"(r[i][14]), "=r"(r[i][15])                               \
                 : "r"(taddr[i])                                                                                \
                 : "memory")
    SSM_TC_LD16(0);
    SSM_TC_LD16(1);
    if constexpr (kBlocks == 4) {
        SSM_TC_LD16(2);
        SSM_TC_LD16(3);
    }
#undef SSM_TC_LD16
    // the registers are written asynchronously: this wait, in a statement that lists them all as in-out
    // operands, keeps every use of them behind it
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0][0]), "+r"(r[0][1]), "+r"(r[0][2]), "+r"(r[0][3]),
                 "+r"(r[0][4]), "+r"(r[0][5]), "+r"(r[0][6]), "+r"(r[0][7]), "+r"(r[0][8]), "+r"(r[0][9]),
                 "+r"(r[0][10]), "+r"(r[0][11]), "+r"(r[0][12]), "+r"(r[0][13]), "+r"(r[0][14]), "+r"(r[0][15])
                 :: "memory");
    asm volatile("" : "+r"(r[1][0]), "+r"(r[1][1]), "+r"(r[1][2]), "+r"(r[1][3]), "+r"(r[1][4]), "+r"(r[1][5]),
                 "+r"(r[1][6]), "+r"(r[1][7]), "+r"(r[1][8]), "+r"(r[1][9]), "+r"(r[1][10]), "+r"(r[1][11]),
                 "+r"(r[1][12]), "+r"(r[1][13]), "+r"(r[1][14]), "+r"(r[1][15]) :: "memory");
    if constexpr (kBlocks == 4) {
        asm volatile("" : "+r"(r[2][0]), "+r"(r[2][1]), "+r"(r[2][2]), "+r"(r[2][3]), "+r"(r[2][4]), "+r"(r[2][5]),
                     "+r"(r[2][6]), "+r"(r[2][7]), "+r"(r[2][8]), "+r"(r[2][9]), "+r"(r[2][10]), "+r"(r[2][11]),
                     "+r"(r[2][12]), "+r"(r[2][13]), "+r"(r[2][14]), "+r"(r[2][15]) :: "memory");
        asm volatile("" : "+r"(r[3][0]), "+r"(r[3][1]), "+r"(r[3][2]), "+r"(r[3][3]), "+r"(r[3][4]), "+r"(r[3][5]),
                     "+r"(r[3][6]), "+r"(r[3][7]), "+r"(r[3][8]), "+r"(r[3][9]), "+r"(r[3][10]), "+r"(r[3][11]),
                     "+r"(r[3][12]), "+r"(r[3][13]), "+r"(r[3][14]), "+r"(r[3][15]) :: "memory");
    }
#pragma unroll
    for (int b = 0; b < kBlocks; ++b)
#pragma unroll
        for (int i = 0; i < 16; ++i) v[b][i] = __uint_as_float(r[b][i]);
}

// byte offset of element (row, k) in a K-major 128-byte-swizzled tile of `rows` rows
__host__ __device__ constexpr uint32_t sw128_offset(int rows, int row, int k) {
    return static_cast<uint32_t>((k >> 6) * rows * 128 + row * 128 + ((((k >> 3) & 7) ^ (row & 7)) << 4) +
                                 ((k & 7) << 1));
}

}  // namespace tc
}  // namespace ssm
