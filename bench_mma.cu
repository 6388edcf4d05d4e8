// tcgen05.mma issue-to-completion time per product on an otherwise idle SM: M = 128, K = 16 bf16 products,
// N = 64 / 128 / 256, accumulating into one TMEM tile (dependent chain) or alternating over two tiles,
// A from shared memory (K-major or MN-major) or from tensor memory.  One CTA per SM, thread 0 issues,
// all waits bounded; every smem / TMEM address stays inside this kernel's own allocation.  The operands are
// zeros: the tensor core's timing does not depend on the values.  Grounds the SSD kernel's notes (its
// products run at about half of these rates, sharing the SM's shared-memory and TMEM bandwidth with the
// element-wise work).
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -I. -o bench_mma bench_mma.cu && ./bench_mma
#include <cstdio>
#include <cstdint>
#include "selective_state_space_156_b300/csrc/tcgen05.cuh"
using namespace ssm;

constexpr int kRep = 32;   // groups of 8 K-steps
__device__ long long g_cycles[148];
__device__ int g_err[148];

template <int N, int kMode>   // 0: A smem K-major, one D; 1: A in TMEM, one D; 2: A smem, two D alternating; 3: A smem MN-major, one D
__global__ void __launch_bounds__(128, 1) mma_bench(int dummy) {
    extern __shared__ __align__(1024) unsigned char sm_raw[];
    const uint32_t raw = smem_u32(sm_raw);
    unsigned char* sm = sm_raw + (((raw + 1023u) & ~1023u) - raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    // A: 128 rows x 128 K (two 16 KB K-blocks); B: 256 rows x 128 K (two 32 KB K-blocks); then barrier + slot
    unsigned char* A = sm;
    unsigned char* B = sm + 32768;
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 32768 + 65536);
    uint32_t* slot = reinterpret_cast<uint32_t*>(sm + 32768 + 65536 + 16);
    for (int i = tid; i < (32768 + 65536) / 16; i += 128) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) { mbar_init(bar, 1); mbar_fence_init(); }
    if (warp == 0) { tc::tmem_alloc(slot, 512); tc::tmem_relinquish(); }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *slot;
    bool ok = true;
    long long cyc = 0;
    if (tid == 0) {
        const uint64_t dA = tc::desc_k_sw128(smem_u32(A)), dB = tc::desc_k_sw128(smem_u32(B));
        const uint64_t dAmn = tc::desc_mn_sw128(smem_u32(B), 32768, 1024);  // B's buffer read MN-major (N x 16 steps)
        const uint32_t id = tc::idesc_bf16(128, N, kMode == 3);
        const long long t0 = clock64();
        for (int r = 0; r < kRep; ++r) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t ka = (ks >> 2) * 16384 + (ks & 3) * 32;
                const uint32_t kb = (ks >> 2) * 32768 + (ks & 3) * 32;
                const uint32_t acc = (r > 0 || ks > 0) ? 1u : 0u;
                if (kMode == 0) tc::mma_bf16(tmem, dA + (ka >> 4), dB + (kb >> 4), id, acc);
                if (kMode == 1) tc::mma_bf16_ts(tmem, tmem + 256 + 8 * ks, dB + (kb >> 4), id, acc);
                if (kMode == 2) tc::mma_bf16(tmem + ((ks & 1) ? 256u : 0u), dA + (ka >> 4), dB + (kb >> 4), id, (r > 0 || ks > 1) ? 1u : 0u);
                if (kMode == 3) tc::mma_bf16(tmem, dAmn + ((ks * 2048) >> 4), dB + (kb >> 4), id, acc);
            }
        }
        tc::mma_commit(bar);
        ok = mbar_wait_bounded(bar, 0);
        cyc = clock64() - t0;
        g_cycles[blockIdx.x] = cyc;
        g_err[blockIdx.x] = ok ? 0 : 1;
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

template <int N, int kMode>
void run(const char* name) {
    auto k = mma_bench<N, kMode>;
    const int smem = 120 * 1024;   // more than half of an SM: one CTA (and one TMEM allocation) per SM
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    k<<<148, 128, smem>>>(0);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) { printf("%s: %s\n", name, cudaGetErrorString(e)); return; }
    long long c[148]; int er[148];
    cudaMemcpyFromSymbol(c, g_cycles, sizeof(c));
    cudaMemcpyFromSymbol(er, g_err, sizeof(er));
    double m = 0; int bad = 0;
    for (int i = 0; i < 148; ++i) { m += c[i]; bad += er[i]; }
    m /= 148;
    const double per = m / (kRep * 8);
    const double flops = 2.0 * 128 * N * 16;
    printf("%-40s %7.1f cycles per product, %6.0f flop/clk/SM%s\n", name, per, flops / per, bad ? " (WAIT TIMED OUT)" : "");
}

int main() {
    run<64, 0>("N=64  A smem K-major, one D");
    run<128, 0>("N=128 A smem K-major, one D");
    run<256, 0>("N=256 A smem K-major, one D");
    run<64, 1>("N=64  A in TMEM, one D");
    run<128, 1>("N=128 A in TMEM, one D");
    run<64, 2>("N=64  A smem, two D alternating");
    run<128, 2>("N=128 A smem, two D alternating");
    run<64, 3>("N=64  A smem MN-major, one D");
    return 0;
}
