// Host side of the tiled bulk-tensor copies: the driver's tensor-map encoder, looked up once through the
// runtime so that the library does not link against libcuda; and the once-per-kernel shared-memory
// attribute of the kernels that use more than 48 KB.
#include <atomic>
#include <cstdlib>
#include <mutex>

#include <cudaTypedefs.h>

#include "ssm_internal.h"
#include "tma.cuh"

namespace ssm {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

bool encode_bf16_map_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t stride_bytes,
                        uint32_t box_inner, uint32_t box_rows) {
    auto fn = encoder();
    if (fn == nullptr) return false;
    if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || stride_bytes % 16 != 0 || (box_inner * 2) % 16 != 0)
        return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_bf16_map_sw128(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box) {
    auto fn = encoder();
    if (fn == nullptr || rank < 2 || rank > 3) return false;
    if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || box[0] * 2 > 128 || (box[0] * 2) % 16 != 0) return false;
    cuuint64_t d[3], st[2];
    cuuint32_t bx[3], es[3];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
    }
    for (int i = 0; i < rank - 1; ++i) {
        if (strides_bytes[i] % 16 != 0) return false;
        st[i] = strides_bytes[i];
    }
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), d, st, bx, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Test hook (ssm_test_withhold_first_copy): set only by the bounded-wait tests, off otherwise.
static std::atomic<int> g_withhold_first_copy{0};

bool withhold_first_copy() { return g_withhold_first_copy.load(std::memory_order_relaxed) != 0; }

}  // namespace ssm

extern "C" SSM_API void ssm_test_withhold_first_copy(int on) {
    ssm::g_withhold_first_copy.store(on ? 1 : 0, std::memory_order_relaxed);
}

namespace ssm {

bool pdl_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("SSM_PDL");
        return !(v != nullptr && v[0] == '0');
    }();
    return on;
}

cudaError_t set_dynamic_smem(const void* kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    struct Key {
        const void* k;
        int bytes, dev;
    };
    static std::mutex mu;
    static Key seen[256];
    static int nseen = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < nseen; ++i)
            if (seen[i].k == kernel && seen[i].bytes == bytes && seen[i].dev == dev) return cudaSuccess;
    }
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (nseen < 256) seen[nseen++] = Key{kernel, bytes, dev};
    return cudaSuccess;
}

cudaError_t resident_blocks(const void* kernel, int threads, int smem_bytes, int* slots) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    struct Key {
        const void* k;
        int threads, smem, dev, slots;
    };
    static std::mutex mu;
    static Key seen[256];
    static int nseen = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < nseen; ++i)
            if (seen[i].k == kernel && seen[i].threads == threads && seen[i].smem == smem_bytes && seen[i].dev == dev) {
                *slots = seen[i].slots;
                return cudaSuccess;
            }
    }
    int sms = 0, per_sm = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem_bytes)) != cudaSuccess)
        return e;
    *slots = sms * per_sm;
    std::lock_guard<std::mutex> lock(mu);
    if (nseen < 256) seen[nseen++] = Key{kernel, threads, smem_bytes, dev, *slots};
    return cudaSuccess;
}

}  // namespace ssm
