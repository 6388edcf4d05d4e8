// Single-token decode step from a constant-size fp32 state cache (B, D, N), updated in place:
// the scan body with L = 1 (datadaily.news "State space models vs Transformer: a practical
// guide", section on how state space models work: h = Abar h + Bbar x_t, y_t = C h + D x_t;
// cache shape (batch, d_inner, d_state) from lshu.cn/news/79586 section 6.5).
// HBM-bound: the state is read and written once per call (2 * B * D * N * 4 bytes).
// With N <= 16 each lane holds at most 4 states; N = 32 and 64 give 8 and 16 per lane.
#include <cstdlib>
#include <cstring>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

constexpr int kDecThreads = 128;
constexpr int kDecLanes = 2;      // lanes per row (64 rows per block)

template <typename T>
__device__ __forceinline__ void load4(const void* base, size_t i, bool vec, float (&v)[4]);
template <>
__device__ __forceinline__ void load4<F32>(const void* base, size_t i, bool vec, float (&v)[4]) {
    const float* p = static_cast<const float*>(base) + i;
    if (vec) {
        const float4 w = __ldg(reinterpret_cast<const float4*>(p));
        v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = __ldg(p + k);
    }
}
template <>
__device__ __forceinline__ void load4<BF16>(const void* base, size_t i, bool vec, float (&v)[4]) {
    const uint16_t* p = static_cast<const uint16_t*>(base) + i;
    if (vec) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
        v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = bf16_to_f32(__ldg(p + k));
    }
}

// Lane e of a row holds the states n = 8k + 4e + i (i < 4, k < NSL / 4): for N = 16 each warp-wide
// 16-byte load or store of the state covers whole 32-byte sectors (the two lanes of a row take the
// two halves of a sector), and every lane keeps 32 bytes of the HBM stream in flight.  A, B and C of
// those states come in with 16-byte (A) and 8-byte (bf16 B, C) loads.  The per-row scalars (dt, v)
// are computed by both lanes; the readout is summed over the two lanes with one shuffle and lane 0
// applies the D skip and the gate.  Zero-order hold as in the scan: h' = Abar (h - ng) + ng with
// ng = -(v / a) B, exact at the fixed point; a == 0 uses the limit dt B.
template <typename T, int NSL, bool kZOH>
__global__ void __launch_bounds__(kDecThreads) state_update_kernel(float* __restrict__ state, const void* __restrict__ u,
                                                                   const void* __restrict__ delta, const float* __restrict__ A,
                                                                   const void* __restrict__ Bm, const void* __restrict__ Cm,
                                                                   const float* __restrict__ Dskip,
                                                                   const float* __restrict__ delta_bias,
                                                                   const void* __restrict__ z, void* __restrict__ y, int D,
                                                                   int N, int softplus_on, int vec) {
    const int e = threadIdx.x & (kDecLanes - 1);
    const int d = blockIdx.x * (kDecThreads / kDecLanes) + threadIdx.x / kDecLanes;
    const bool active = d < D;
    const int b = blockIdx.y;
    const size_t row = (size_t)b * D + (active ? d : 0);

    // issue every load first: the state (the HBM stream), then the L2-resident operands
    float h[NSL], av[NSL], Bt[NSL], Ct[NSL];
#pragma unroll
    for (int k = 0; k < NSL / 4; ++k) {
        const int n0 = 4 * kDecLanes * k + 4 * e;
        const bool full = vec && active && n0 + 3 < N;
        if (full) {
            const float4 w = __ldcs(reinterpret_cast<const float4*>(state + row * N + n0));
            h[4 * k] = w.x; h[4 * k + 1] = w.y; h[4 * k + 2] = w.z; h[4 * k + 3] = w.w;
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) h[4 * k + i] = (active && n0 + i < N) ? state[row * N + n0 + i] : 0.0f;
        }
        float t4[4];
        if (full) {
            load4<F32>(A, (size_t)d * N + n0, true, t4);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) t4[i] = (active && n0 + i < N) ? __ldg(A + (size_t)d * N + n0 + i) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) av[4 * k + i] = t4[i];
        if (full) {
            load4<T>(Bm, (size_t)b * N + n0, true, t4);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) t4[i] = (n0 + i < N) ? load1<T>(Bm, (size_t)b * N + n0 + i) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) Bt[4 * k + i] = t4[i];
        if (full) {
            load4<T>(Cm, (size_t)b * N + n0, true, t4);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) t4[i] = (n0 + i < N) ? load1<T>(Cm, (size_t)b * N + n0 + i) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) Ct[4 * k + i] = t4[i];
    }
    const float uv = active ? load1<T>(u, row) : 0.0f;
    const float s = (active ? load1<T>(delta, row) : 0.0f) + ((delta_bias != nullptr && active) ? __ldg(delta_bias + d) : 0.0f);
    const float dt = softplus_on ? softplus(s) : s;

    float yp = 0.0f;
#pragma unroll
    for (int i = 0; i < NSL; ++i) {
        const float a = av[i];
        const float ab = ex2(dt * (a * kLog2e));
        if (kZOH) {
            if (a != 0.0f) {
                const float ng = (uv * -rcp(a)) * Bt[i];
                h[i] = fmaf(ab, h[i] - ng, ng);
            } else {
                h[i] = fmaf(dt * uv, Bt[i], h[i]);  // the a -> 0 limit: Abar = 1, Bbar = dt B
            }
        } else {
            h[i] = fmaf(ab, h[i], (dt * uv) * Bt[i]);
        }
        yp = fmaf(Ct[i], h[i], yp);
    }
#pragma unroll
    for (int m = 1; m < kDecLanes; m <<= 1) yp += __shfl_xor_sync(0xffffffffu, yp, m);
    if (!active) return;
    if (e == 0) {
        const float gate = z != nullptr ? silu(load1<T>(z, row)) : 1.0f;
        const float dsk = Dskip != nullptr ? __ldg(Dskip + d) : 0.0f;
        store1<T>(y, row, fmaf(dsk, uv, yp) * gate);
    }
#pragma unroll
    for (int k = 0; k < NSL / 4; ++k) {
        const int n0 = 4 * kDecLanes * k + 4 * e;
        if (vec && n0 + 3 < N) {
            __stcs(reinterpret_cast<float4*>(state + row * N + n0),
                   make_float4(h[4 * k], h[4 * k + 1], h[4 * k + 2], h[4 * k + 3]));
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (n0 + i < N) state[row * N + n0 + i] = h[4 * k + i];
        }
    }
}

template <typename T, int NSL>
static cudaError_t launch_su_ns(float* state, const void* u, const void* delta, const float* A, const void* Bm,
                                const void* Cm, const float* Dskip, const float* delta_bias, const void* z, void* y,
                                int Bsz, int D, int N, int softplus_on, int zoh, cudaStream_t stream) {
    // vector loads need every lane's first state aligned: N % 4 == 0 and aligned bases (16 bytes for the
    // fp32 state and A, 4 elements for B and C)
    const int esz = sizeof(typename T::storage);
    const int vec_state = (N % 4 == 0) && ((reinterpret_cast<uintptr_t>(state) & 15) == 0) &&
                          ((reinterpret_cast<uintptr_t>(A) & 15) == 0) &&
                          ((reinterpret_cast<uintptr_t>(Bm) & (4 * esz - 1)) == 0) &&
                          ((reinterpret_cast<uintptr_t>(Cm) & (4 * esz - 1)) == 0);
    dim3 block(kDecThreads);
    dim3 grid((unsigned)((D + kDecThreads / kDecLanes - 1) / (kDecThreads / kDecLanes)), (unsigned)Bsz);
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
    // states per lane: N / kDecLanes rounded up to a multiple of 4
    if (N <= 8) return launch_su_ns<T, 4>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
    if (N <= 16) return launch_su_ns<T, 8>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
    if (N <= 32) return launch_su_ns<T, 16>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
    return launch_su_ns<T, 32>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
}

// SSM_DECODE_KERNEL=rows keeps every call on the row kernel above (for comparisons); by default calls
// that meet its requirements take the streamed kernel of state_update_bulk.cu.
static bool bulk_decode_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("SSM_DECODE_KERNEL");
        return !(v != nullptr && std::strcmp(v, "rows") == 0);
    }();
    return on;
}

cudaError_t launch_state_update(float* state, const void* u, const void* delta, const float* A, const void* Bm,
                                const void* Cm, const float* Dskip, const float* delta_bias, const void* z, void* y,
                                int Bsz, int D, int N, int softplus_on, int zoh, int dtype, cudaStream_t stream) {
    if (bulk_decode_enabled() && state_update_bulk_eligible(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, D, N))
        return launch_state_update_bulk(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh,
                                        dtype, stream);
    if (dtype == 1)
        return launch_su_t<BF16>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
    return launch_su_t<F32>(state, u, delta, A, Bm, Cm, Dskip, delta_bias, z, y, Bsz, D, N, softplus_on, zoh, stream);
}

}  // namespace ssm
