// Single-token decode step from a constant-size fp32 state cache (B, D, N), updated in place:
// the scan body with L = 1 (datadaily.news "State space models vs Transformer: a practical
// guide", section on how state space models work: h = Abar h + Bbar x_t, y_t = C h + D x_t;
// cache shape (batch, d_inner, d_state) from lshu.cn/news/79586 section 6.5).
// HBM-bound: the state is read and written once per call (2 * B * D * N * 4 bytes).
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

constexpr int kDecThreads = 128;

template <typename T, int NS, bool kZOH>
__global__ void __launch_bounds__(kDecThreads) state_update_kernel(float* __restrict__ state, const void* __restrict__ u,
                                                                   const void* __restrict__ delta, const float* __restrict__ A,
                                                                   const void* __restrict__ Bm, const void* __restrict__ Cm,
                                                                   const float* __restrict__ Dskip,
                                                                   const float* __restrict__ delta_bias,
                                                                   const void* __restrict__ z, void* __restrict__ y, int D,
                                                                   int N, int softplus_on, int vec_state) {
    const int d = blockIdx.x * kDecThreads + threadIdx.x;
    if (d >= D) return;
    const int b = blockIdx.y;
    const size_t row = (size_t)b * D + d;

    float h[NS];
    if (vec_state) {
        const float4* p = reinterpret_cast<const float4*>(state + row * NS);
#pragma unroll
        for (int q = 0; q < NS / 4; ++q) {
            float4 v = p[q];
            h[4 * q] = v.x; h[4 * q + 1] = v.y; h[4 * q + 2] = v.z; h[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int n = 0; n < NS; ++n) h[n] = n < N ? state[row * N + n] : 0.0f;
    }

    const float uv = load1<T>(u, row);
    const float s = load1<T>(delta, row) + (delta_bias != nullptr ? __ldg(delta_bias + d) : 0.0f);
    const float dt = softplus_on ? softplus(s) : s;
    const float gate = z != nullptr ? silu(load1<T>(z, row)) : 1.0f;

    float y0 = 0.0f, y1 = 0.0f;
#pragma unroll
    for (int n = 0; n < NS; ++n) {
        if (n >= N) break;
        const float av = __ldg(A + (size_t)d * N + n);
        const float Bt = load1<T>(Bm, (size_t)b * N + n);
        const float Ct = load1<T>(Cm, (size_t)b * N + n);
        const float ab = ex2(dt * av * kLog2e);
        float bb;
        if (kZOH)
            bb = av != 0.0f ? (ab - 1.0f) * (1.0f / av) : dt;   // limit dt at a = 0
        else
            bb = dt;
        h[n] = fmaf(ab, h[n], bb * Bt * uv);
        if (n & 1) y1 = fmaf(Ct, h[n], y1);
        else y0 = fmaf(Ct, h[n], y0);
    }
    const float dsk = Dskip != nullptr ? __ldg(Dskip + d) : 0.0f;
    store1<T>(y, row, fmaf(dsk, uv, y0 + y1) * gate);

    if (vec_state) {
        float4* p = reinterpret_cast<float4*>(state + row * NS);
#pragma unroll
        for (int q = 0; q < NS / 4; ++q) p[q] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
    } else {
#pragma unroll
        for (int n = 0; n < NS; ++n)
            if (n < N) state[row * N + n] = h[n];
    }
}

template <typename T, int NS>
static cudaError_t launch_su_ns(float* state, const void* u, const void* delta, const float* A, const void* Bm,
                                const void* Cm, const float* Dskip, const float* delta_bias, const void* z, void* y,
                                int Bsz, int D, int N, int softplus_on, int zoh, cudaStream_t stream) {
    const int vec_state = (N == NS) && ((reinterpret_cast<uintptr_t>(state) & 15) == 0);
    dim3 block(kDecThreads);
    dim3 grid((unsigned)((D + kDecThreads - 1) / kDecThreads), (unsigned)Bsz);
    if (zoh)
        state_update_kernel<T, NS, true><<<grid, block, 0, stream>>>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, D,
                                                                     N, softplus_on, vec_state);
    else
        state_update_kernel<T, NS, false><<<grid, block, 0, stream>>>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y,
                                                                      D, N, softplus_on, vec_state);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_su_t(float* state, const void* u, const void* delta, const float* A, const void* Bm,
                               const void* Cm, const float* Dskip, const float* delta_bias, const void* z, void* y,
                               int Bsz, int D, int N, int softplus_on, int zoh, cudaStream_t stream) {
    if (N <= 4) return launch_su_ns<T, 4>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
    if (N <= 8) return launch_su_ns<T, 8>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
    if (N <= 16) return launch_su_ns<T, 16>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
    if (N <= 32) return launch_su_ns<T, 32>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
    return launch_su_ns<T, 64>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
}

cudaError_t launch_state_update(float* state, const void* u, const void* delta, const float* A, const void* Bm,
                                const void* Cm, const float* Dskip, const float* delta_bias, const void* z, void* y,
                                int Bsz, int D, int N, int softplus_on, int zoh, int dtype, cudaStream_t stream) {
    if (dtype == 1)
        return launch_su_t<BF16>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
    return launch_su_t<F32>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
}

}  // namespace ssm
