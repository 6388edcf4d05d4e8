// Per-SM-per-clock issue rates of the MUFU (ex2, rcp, lg2, tanh) and FP32 FMA pipes (scalar fma and packed
// fma.rn.f32x2, the latter as lane operations), measured with
// clock64 inside the kernel so the result does not depend on the SM clock.  bench.py builds and runs
// it to ground the ALU roofline of the scan kernels (peak = rate/clk/SM x SMs x max SM clock).
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o bench_peaks bench_peaks.cu && ./bench_peaks
// Prints one JSON object.  Every launch touches only its own buffers, in bounds; no waits.
#include <cstdio>
#include <cstdlib>
#include <vector>
#include <cuda_runtime.h>

#define CK(x)                                                                                   \
    do {                                                                                        \
        cudaError_t e_ = (x);                                                                   \
        if (e_ != cudaSuccess) {                                                                \
            printf("{\"error\": \"%s at line %d\"}\n", cudaGetErrorString(e_), __LINE__);      \
            exit(1);                                                                            \
        }                                                                                       \
    } while (0)

template <int OP>
__device__ __forceinline__ float op(float x) {
    float y;
    if (OP == 0) asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    if (OP == 1) {  // x -> 1 / (x + 1): the add keeps the chain from folding to the identity
        float t;
        asm volatile("add.f32 %0, %1, 0f3F800000;" : "=f"(t) : "f"(x));
        asm volatile("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(t));
    }
    if (OP == 2) asm volatile("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    if (OP == 3) asm volatile("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    if (OP == 4) asm volatile("fma.rn.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(x), "f"(0.99991f), "f"(1e-4f));
    return y;
}

// Packed pair: one fma.rn.f32x2 on (x, x + 1) per call, counted as two lane operations.
__device__ __forceinline__ unsigned long long op_pair(unsigned long long x) {
    unsigned long long y, m, c;
    asm volatile("mov.b64 %0, {%1, %2};" : "=l"(m) : "f"(0.99991f), "f"(0.99993f));
    asm volatile("mov.b64 %0, {%1, %2};" : "=l"(c) : "f"(1e-4f), "f"(2e-4f));
    asm volatile("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(y) : "l"(x), "l"(m), "l"(c));
    return y;
}

// 8 independent chains of packed pairs per thread (16 lane operations per iteration).
__global__ void __launch_bounds__(512) rate_pair_kernel(float* out, int iters, long long* cyc) {
    unsigned long long v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float a = 1.0f + 0.001f * (threadIdx.x & 31) + 0.01f * j;
        asm volatile("mov.b64 %0, {%1, %2};" : "=l"(v[j]) : "f"(a), "f"(a + 0.5f));
    }
    __syncthreads();
    long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = op_pair(v[j]);
    }
    long long t1 = clock64();
    __syncthreads();
    if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float a, b;
        asm volatile("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v[j]));
        s += a + b;
    }
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// 8 independent dependency chains per thread; the volatile asm keeps every operation.
template <int OP>
__global__ void __launch_bounds__(512) rate_kernel(float* out, int iters, long long* cyc) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 1.0f + 0.001f * (threadIdx.x & 31) + 0.01f * j;
    __syncthreads();
    long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = op<OP>(v[j]);
    }
    long long t1 = clock64();
    __syncthreads();
    if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += v[j];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

template <int OP>
double rate(int sms) {
    const int threads = 512, blocks = sms * 2, iters = 2048;  // 2 x 512 threads resident per SM
    float* out;
    long long* cyc;
    CK(cudaMalloc(&out, sizeof(float) * threads * blocks));
    CK(cudaMalloc(&cyc, sizeof(long long) * blocks));
    if constexpr (OP == 5) {
        rate_pair_kernel<<<blocks, threads>>>(out, 8, cyc);
        CK(cudaDeviceSynchronize());
        rate_pair_kernel<<<blocks, threads>>>(out, iters, cyc);
    } else {
        rate_kernel<OP><<<blocks, threads>>>(out, 8, cyc);
        CK(cudaDeviceSynchronize());
        rate_kernel<OP><<<blocks, threads>>>(out, iters, cyc);
    }
    CK(cudaDeviceSynchronize());
    std::vector<long long> c(blocks);
    CK(cudaMemcpy(c.data(), cyc, sizeof(long long) * blocks, cudaMemcpyDeviceToHost));
    double cmax = 0;
    for (long long x : c) cmax = cmax > (double)x ? cmax : (double)x;
    CK(cudaFree(out));
    CK(cudaFree(cyc));
    // both blocks of an SM run at the same time, so an SM retires 2 * threads * iters * 8 ops in cmax clocks
    // (the packed probe: two lane operations per op)
    return (OP == 5 ? 2.0 : 1.0) * 2.0 * threads * iters * 8.0 / cmax;
}

int main() {
    int dev = 0, sms = 0, clk = 0;
    CK(cudaGetDevice(&dev));
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    CK(cudaDeviceGetAttribute(&clk, cudaDevAttrClockRate, dev));
    int occ = 0;
    CK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, rate_kernel<4>, 512, 0));
    if (occ < 2) {
        printf("{\"error\": \"fewer than 2 probe blocks fit on an SM\"}\n");
        return 1;
    }
    double ex2 = rate<0>(sms), rcp = rate<1>(sms), lg2 = rate<2>(sms), th = rate<3>(sms), fma = rate<4>(sms);
    double fma2 = rate<5>(sms);
    printf("{\"sms\": %d, \"max_sm_mhz\": %.0f, \"per_clk_per_sm\": {\"ex2\": %.2f, \"rcp\": %.2f, \"lg2\": %.2f, "
           "\"tanh\": %.2f, \"ffma\": %.2f, \"ffma2_lanes\": %.2f}}\n",
           sms, clk / 1000.0, ex2, rcp, lg2, th, fma, fma2);
    return 0;
}
