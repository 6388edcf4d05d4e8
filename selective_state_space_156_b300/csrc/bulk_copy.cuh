// Shared-memory mbarriers and 1-D bulk copies (the TMA engine without a tensor map), as inline PTX for
// sm_90 and later.  A copy moves a contiguous global range into shared memory and signals completion
// by decrementing the transaction count of an mbarrier; a consumer waits on the barrier's phase.
// Both addresses must be 16-byte aligned and the size a multiple of 16 bytes (callers check).
//
// Every wait is bounded: mbar_wait_bounded gives up after about kWaitLimitCycles SM clocks and returns
// false, so a kernel can record the failure and return instead of spinning forever.
#pragma once

#include <cstdint>

namespace ssm {

constexpr long long kWaitLimitCycles = 1ll << 31;  // about one second at 2 GHz

__device__ __forceinline__ unsigned smem_u32(const void* p) {
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// make the initialised barriers visible to the async proxy (the bulk-copy engine)
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// one arrival that also raises the barrier's expected transaction bytes
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// a plain arrival (release semantics: this thread's earlier shared-memory reads are done)
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
    unsigned done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// true once the phase with the given parity has completed; false after the wait limit
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitLimitCycles) return false;
    }
    return true;
}

// Programmatic dependent launch: a kernel launched with programmatic stream serialization may start
// while the previous kernel of the stream drains; pdl_wait blocks until that kernel has completed and
// its memory is visible (kernels call it before their first global access), pdl_release lets the next
// such kernel be scheduled.  Both are no-ops for a plain launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// global -> shared bulk copy completing on `bar` (the CTA's own shared memory)
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

}  // namespace ssm
