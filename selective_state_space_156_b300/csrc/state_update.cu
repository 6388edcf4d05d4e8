// Single-token decode step from a constant-size fp32 state cache (B, D, N), updated in place:
// the scan body with L = 1 (datadaily.news "State space models vs Transformer: a practical
// guide", section on how state space models work: h = Abar h + Bbar x_t, y_t = C h + D x_t;
// cache shape (batch, d_inner, d_state) from lshu.cn/news/79586 section 6.5).
// HBM-bound: the state is read and written once per call (2 * B * D * N * 4 bytes).
// With N <= 16 each lane holds at most 4 states; N = 32 and 64 give 8 and 16 per lane.
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

constexpr int kDecThreads = 128;  // 32 rows x 4 lanes

// Lane q of a row holds the states n = 16k + 4q + i (i < 4, k < NSL / 4): for N = 16 the four lanes of
// a row hold 64 contiguous bytes, so a warp's 16-byte loads and stores cover 512 contiguous bytes of
// the state cache.  The per-row scalars (dt, v, gate) are computed by all four lanes; the readout is
// reduced over the four lanes with two shuffles.
template <typename T, int NSL, bool kZOH>
__global__ void __launch_bounds__(kDecThreads) state_update_kernel(float* __restrict__ state, const void* __restrict__ u,
                                                                   const void* __restrict__ delta, const float* __restrict__ A,
                                                                   const void* __restrict__ Bm, const void* __restrict__ Cm,
                                                                   const float* __restrict__ Dskip,
                                                                   const float* __restrict__ delta_bias,
                                                                   const void* __restrict__ z, void* __restrict__ y, int D,
                                                                   int N, int softplus_on, int vec_state) {
    const int q = threadIdx.x & 3;
    const int d = blockIdx.x * (kDecThreads / 4) + (threadIdx.x >> 2);
    const bool active = d < D;
    const int b = blockIdx.y;
    const size_t row = (size_t)b * D + (active ? d : 0);

    float h[NSL];
    if (vec_state) {
#pragma unroll
        for (int k = 0; k < NSL / 4; ++k) {
            const int n0 = 16 * k + 4 * q;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (active && n0 < N) v = __ldcs(reinterpret_cast<const float4*>(state + row * N + n0));
            h[4 * k] = v.x; h[4 * k + 1] = v.y; h[4 * k + 2] = v.z; h[4 * k + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < NSL / 4; ++k)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int n = 16 * k + 4 * q + i;
                h[4 * k + i] = (active && n < N) ? state[row * N + n] : 0.0f;
            }
    }

    const float uv = active ? load1<T>(u, row) : 0.0f;
    const float s = (active ? load1<T>(delta, row) : 0.0f) + ((delta_bias != nullptr && active) ? __ldg(delta_bias + d) : 0.0f);
    const float dt = softplus_on ? softplus(s) : s;

    float yp = 0.0f;
#pragma unroll
    for (int k = 0; k < NSL / 4; ++k)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int n = 16 * k + 4 * q + i;
            if (!active || n >= N) continue;
            const float av = __ldg(A + (size_t)d * N + n);
            const float Bt = load1<T>(Bm, (size_t)b * N + n);
            const float Ct = load1<T>(Cm, (size_t)b * N + n);
            const float ab = ex2(dt * av * kLog2e);
            float bb;
            if (kZOH)
                bb = av != 0.0f ? (ab - 1.0f) * (1.0f / av) : dt;  // limit dt at a = 0
            else
                bb = dt;
            float& hn = h[4 * k + i];
            hn = fmaf(ab, hn, bb * Bt * uv);
            yp = fmaf(Ct, hn, yp);
        }
    yp += __shfl_xor_sync(0xffffffffu, yp, 1);
    yp += __shfl_xor_sync(0xffffffffu, yp, 2);
    if (!active) return;
    if (q == 0) {
        const float gate = z != nullptr ? silu(load1<T>(z, row)) : 1.0f;
        const float dsk = Dskip != nullptr ? __ldg(Dskip + d) : 0.0f;
        store1<T>(y, row, fmaf(dsk, uv, yp) * gate);
    }
    if (vec_state) {
#pragma unroll
        for (int k = 0; k < NSL / 4; ++k) {
            const int n0 = 16 * k + 4 * q;
            if (n0 < N)
                __stcs(reinterpret_cast<float4*>(state + row * N + n0),
                       make_float4(h[4 * k], h[4 * k + 1], h[4 * k + 2], h[4 * k + 3]));
        }
    } else {
#pragma unroll
        for (int k = 0; k < NSL / 4; ++k)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int n = 16 * k + 4 * q + i;
                if (n < N) state[row * N + n] = h[4 * k + i];
            }
    }
}

template <typename T, int NSL>
static cudaError_t launch_su_ns(float* state, const void* u, const void* delta, const float* A, const void* Bm,
                                const void* Cm, const float* Dskip, const float* delta_bias, const void* z, void* y,
                                int Bsz, int D, int N, int softplus_on, int zoh, cudaStream_t stream) {
    // 16-byte vectors need every lane's first state 16-byte aligned: N % 4 == 0 and an aligned base
    const int vec_state = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(state) & 15) == 0);
    dim3 block(kDecThreads);
    dim3 grid((unsigned)((D + kDecThreads / 4 - 1) / (kDecThreads / 4)), (unsigned)Bsz);
    if (zoh)
        state_update_kernel<T, NSL, true><<<grid, block, 0, stream>>>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, D,
                                                                      N, softplus_on, vec_state);
    else
        state_update_kernel<T, NSL, false><<<grid, block, 0, stream>>>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y,
                                                                       D, N, softplus_on, vec_state);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_su_t(float* state, const void* u, const void* delta, const float* A, const void* Bm,
                               const void* Cm, const float* Dskip, const float* delta_bias, const void* z, void* y,
                               int Bsz, int D, int N, int softplus_on, int zoh, cudaStream_t stream) {
    if (N <= 16) return launch_su_ns<T, 4>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
    if (N <= 32) return launch_su_ns<T, 8>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
    return launch_su_ns<T, 16>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
}

cudaError_t launch_state_update(float* state, const void* u, const void* delta, const float* A, const void* Bm,
                                const void* Cm, const float* Dskip, const float* delta_bias, const void* z, void* y,
                                int Bsz, int D, int N, int softplus_on, int zoh, int dtype, cudaStream_t stream) {
    if (dtype == 1)
        return launch_su_t<BF16>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
    return launch_su_t<F32>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
}

}  // namespace ssm
