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
// applies the D skip and the gate.  Zero-order hold in the exact form h' = Abar h + E v B, with
// E = (exp(dt a) - 1) / a from zoh_factor (a Taylor series where |dt a| is small, dt at a = 0).
template <typename T, int NSL, bool kZOH, bool kConv>
__global__ void __launch_bounds__(kDecThreads) state_update_kernel(const DecodeStep s, int vec) {
    float* __restrict__ state = s.state;
    const int D = s.D, N = s.N;
    const int e = threadIdx.x & (kDecLanes - 1);
    const int d = blockIdx.x * (kDecThreads / kDecLanes) + threadIdx.x / kDecLanes;
    const bool active = d < D;
    const int b = blockIdx.y;
    const size_t row = (size_t)b * D + (active ? d : 0);  // u, delta, z, y
    // the row's slot in the state cache (state_indices), negative for a padding row
    const int slot = s.state_indices != nullptr ? __ldg(s.state_indices + b) : b;
    if (slot < 0) {
        if (active && e == 0) store1<T>(s.y, row, 0.0f);
        return;  // uniform over the row's lanes: no shuffle is left half-done
    }
    const size_t srow = (size_t)slot * D + (active ? d : 0);  // state, conv_state

    // issue every load first: the state (the HBM stream), then the L2-resident operands
    float h[NSL], av[NSL], Bt[NSL], Ct[NSL];
#pragma unroll
    for (int k = 0; k < NSL / 4; ++k) {
        const int n0 = 4 * kDecLanes * k + 4 * e;
        const bool full = vec && active && n0 + 3 < N;
        if (full) {
            const float4 w = __ldcs(reinterpret_cast<const float4*>(state + srow * N + n0));
            h[4 * k] = w.x; h[4 * k + 1] = w.y; h[4 * k + 2] = w.z; h[4 * k + 3] = w.w;
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) h[4 * k + i] = (active && n0 + i < N) ? state[srow * N + n0 + i] : 0.0f;
        }
        float t4[4];
        if (full) {
            load4<F32>(s.A, (size_t)d * N + n0, true, t4);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) t4[i] = (active && n0 + i < N) ? __ldg(s.A + (size_t)d * N + n0 + i) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) av[4 * k + i] = t4[i];
        if (full) {
            load4<T>(s.Bm, (size_t)b * N + n0, true, t4);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) t4[i] = (n0 + i < N) ? load1<T>(s.Bm, (size_t)b * N + n0 + i) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) Bt[4 * k + i] = t4[i];
        if (full) {
            load4<T>(s.Cm, (size_t)b * N + n0, true, t4);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) t4[i] = (n0 + i < N) ? load1<T>(s.Cm, (size_t)b * N + n0 + i) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) Ct[4 * k + i] = t4[i];
    }
    float uv = active ? load1<T>(s.x, row) : 0.0f;
    if (kConv) {
        // v = SiLU(conv_b + sum_k w_k x_{t-W+1+k}) with x before t from the row's conv state (oldest
        // first); both lanes of the row read the state before lane 0 writes the shifted one back
        using Sx = typename T::storage;
        const int W = s.conv_width, W1 = W - 1;
        Sx* cs = static_cast<Sx*>(s.conv_state) + srow * W1;
        float c = (s.conv_b != nullptr && active) ? __ldg(s.conv_b + d) : 0.0f;
        Sx hist[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            hist[k] = (active && k < W1) ? cs[k] : Sx(0);  // plain loads: this kernel writes the state back
            float hv;
            if constexpr (T::kBytes == 2) hv = bf16_to_f32(hist[k]);
            else hv = hist[k];
            if (active && k < W1) c = fmaf(__ldg(s.conv_w + (size_t)d * W + k), hv, c);
        }
        if (active) c = fmaf(__ldg(s.conv_w + (size_t)d * W + W1), uv, c);
        __syncwarp();
        if (active && e == 0) {
            const Sx xraw = static_cast<const Sx*>(s.x)[row];
#pragma unroll
            for (int k = 0; k < 3; ++k)
                if (k < W1) cs[k] = k + 1 < W1 ? hist[k + 1] : xraw;
        }
        uv = silu(c);
    }
    const float sr = (active ? load1<T>(s.delta, row) : 0.0f) +
                     ((s.delta_bias != nullptr && active) ? __ldg(s.delta_bias + d) : 0.0f);
    const float dt = s.softplus ? softplus(sr) : sr;

    float yp = 0.0f;
#pragma unroll
    for (int i = 0; i < NSL; ++i) {
        const float a = av[i];
        const float y = dt * (a * kLog2e);
        if (kZOH) {  // exact form: E (and Abar) from the series where |dt a| < 2^-4, dt at a = 0
            float ab;
            const float E = zoh_exact(dt, y, a != 0.0f ? rcp(a) : 0.0f, ab);
            h[i] = fmaf(ab, h[i], E * (uv * Bt[i]));
        } else {
            h[i] = fmaf(abar_exact(y), h[i], (dt * uv) * Bt[i]);
        }
        yp = fmaf(Ct[i], h[i], yp);
    }
#pragma unroll
    for (int m = 1; m < kDecLanes; m <<= 1) yp += __shfl_xor_sync(0xffffffffu, yp, m);
    if (!active) return;
    if (e == 0) {
        const float gate = s.z != nullptr ? silu(load1<T>(s.z, row)) : 1.0f;
        const float dsk = s.Dskip != nullptr ? __ldg(s.Dskip + d) : 0.0f;
        store1<T>(s.y, row, fmaf(dsk, uv, yp) * gate);
    }
#pragma unroll
    for (int k = 0; k < NSL / 4; ++k) {
        const int n0 = 4 * kDecLanes * k + 4 * e;
        if (vec && n0 + 3 < N) {
            __stcs(reinterpret_cast<float4*>(state + srow * N + n0),
                   make_float4(h[4 * k], h[4 * k + 1], h[4 * k + 2], h[4 * k + 3]));
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (n0 + i < N) state[srow * N + n0 + i] = h[4 * k + i];
        }
    }
}

template <typename T, int NSL>
static cudaError_t launch_su_ns(const DecodeStep& s, cudaStream_t stream) {
    // vector loads need every lane's first state aligned: N % 4 == 0 and aligned bases (16 bytes for the
    // fp32 state and A, 4 elements for B and C)
    const int esz = sizeof(typename T::storage);
    const int vec_state = (s.N % 4 == 0) && ((reinterpret_cast<uintptr_t>(s.state) & 15) == 0) &&
                          ((reinterpret_cast<uintptr_t>(s.A) & 15) == 0) &&
                          ((reinterpret_cast<uintptr_t>(s.Bm) & (4 * esz - 1)) == 0) &&
                          ((reinterpret_cast<uintptr_t>(s.Cm) & (4 * esz - 1)) == 0);
    dim3 block(kDecThreads);
    dim3 grid((unsigned)((s.D + kDecThreads / kDecLanes - 1) / (kDecThreads / kDecLanes)), (unsigned)s.Bsz);
    const bool conv = s.conv_w != nullptr;
    if (s.zoh) {
        if (conv) state_update_kernel<T, NSL, true, true><<<grid, block, 0, stream>>>(s, vec_state);
        else state_update_kernel<T, NSL, true, false><<<grid, block, 0, stream>>>(s, vec_state);
    } else {
        if (conv) state_update_kernel<T, NSL, false, true><<<grid, block, 0, stream>>>(s, vec_state);
        else state_update_kernel<T, NSL, false, false><<<grid, block, 0, stream>>>(s, vec_state);
    }
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_su_t(const DecodeStep& s, cudaStream_t stream) {
    // states per lane: N / kDecLanes rounded up to a multiple of 4
    if (s.N <= 8) return launch_su_ns<T, 4>(s, stream);
    if (s.N <= 16) return launch_su_ns<T, 8>(s, stream);
    if (s.N <= 32) return launch_su_ns<T, 16>(s, stream);
    return launch_su_ns<T, 32>(s, stream);
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

cudaError_t launch_state_update(const DecodeStep& s, cudaStream_t stream) {
    if (bulk_decode_enabled() && state_update_bulk_eligible(s)) return launch_state_update_bulk(s, stream);
    if (s.dtype == 1) return launch_su_t<BF16>(s, stream);
    return launch_su_t<F32>(s, stream);
}

}  // namespace ssm
