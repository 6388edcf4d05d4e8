// Standalone causal depthwise conv1d (+ optional SiLU): the front end of the Mamba block
// (dpshk.com/news/3333417 section 5.2: Conv1d with padding width-1, groups = channels, output
// cropped to the first L steps, then SiLU).  Tap k of a width-W filter multiplies x_{t-W+1+k}.
// HBM-bound: one read of x and one write of y.
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

constexpr int kConvThreads = 128;
constexpr int kConvTile = 512;  // timesteps per thread

template <typename T>
__global__ void __launch_bounds__(kConvThreads) causal_conv1d_kernel(const void* __restrict__ x, const float* __restrict__ w,
                                                                     const float* __restrict__ bias, void* __restrict__ y,
                                                                     int D, int L, int W, int silu_on, int vec) {
    const int d = blockIdx.x * kConvThreads + threadIdx.x;
    if (d >= D) return;
    const size_t row = (size_t)blockIdx.y * D + d;
    const size_t rowoff = row * (size_t)L;
    const int t0 = blockIdx.z * kConvTile;
    const int t1 = min(L, t0 + kConvTile);

    float wk[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < 4; ++i)  // tap i of the 4-wide window is tap i - (4 - W) of the filter
        wk[i] = i >= 4 - W ? __ldg(w + (size_t)d * W + i - (4 - W)) : 0.0f;
    const float cb = bias != nullptr ? __ldg(bias + d) : 0.0f;
    float xh[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const int t = t0 - 3 + k;
        xh[k] = t >= 0 ? load1<T>(x, rowoff + t) : 0.0f;
    }

    for (int tg = t0; tg < t1; tg += 8) {
        const int nv = min(8, t1 - tg);
        float xv[8], out[8];
        if (vec && nv == 8) {
            load8<T>(x, rowoff + tg, xv);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) xv[j] = j < nv ? load1<T>(x, rowoff + tg + j) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float acc = fmaf(wk[0], xh[0], cb);
            acc = fmaf(wk[1], xh[1], acc);
            acc = fmaf(wk[2], xh[2], acc);
            acc = fmaf(wk[3], xv[j], acc);
            xh[0] = xh[1];
            xh[1] = xh[2];
            xh[2] = xv[j];
            out[j] = silu_on ? silu(acc) : acc;
        }
        if (vec && nv == 8) {
            store8<T>(y, rowoff + tg, out);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < nv) store1<T>(y, rowoff + tg + j, out[j]);
        }
    }
}

cudaError_t launch_causal_conv1d(const void* x, const float* w, const float* b, void* y, int Bsz, int D, int L, int width,
                                 int silu_on, int dtype, cudaStream_t stream) {
    const int esize = dtype == 1 ? 2 : 4;
    const int vec = (((size_t)L * esize) % 16 == 0) && ((reinterpret_cast<uintptr_t>(x) & 15) == 0) &&
                    ((reinterpret_cast<uintptr_t>(y) & 15) == 0);
    dim3 block(kConvThreads);
    dim3 grid((unsigned)((D + kConvThreads - 1) / kConvThreads), (unsigned)Bsz, (unsigned)((L + kConvTile - 1) / kConvTile));
    if (dtype == 1)
        causal_conv1d_kernel<BF16><<<grid, block, 0, stream>>>(x, w, b, y, D, L, width, silu_on, vec);
    else
        causal_conv1d_kernel<F32><<<grid, block, 0, stream>>>(x, w, b, y, D, L, width, silu_on, vec);
    return cudaGetLastError();
}

// The conv history a later call needs: the last W1 = conv_width - 1 inputs of every row, reaching back
// into the row's previous history when L < W1 (a chunked prefill or the first decode steps carry it
// on; dpshk.com/news/5205047 section 1.3).  One thread per row; each thread reads all its sources
// (plain loads: the history may be the output buffer) before it writes.
template <typename T>
__global__ void __launch_bounds__(kConvThreads) conv_history_kernel(const void* __restrict__ x, const void* conv_init,
                                                                    void* conv_final, const int* state_indices, int D,
                                                                    int L, int W1) {
    using S = typename T::storage;
    const int d = blockIdx.x * kConvThreads + threadIdx.x, b = blockIdx.y;
    if (d >= D) return;
    const int slot = state_indices != nullptr ? state_indices[b] : b;
    if (slot < 0) return;  // a padding row owns no slot
    const size_t r = (size_t)b * D + d, sr = (size_t)slot * D + d;
    const S* xr = static_cast<const S*>(x) + r * (size_t)L;
    const S* hi = conv_init != nullptr ? static_cast<const S*>(conv_init) + sr * W1 : nullptr;
    S v[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const int t = L - W1 + i;
        v[i] = S(0);
        if (i < W1) v[i] = t >= 0 ? xr[t] : (hi != nullptr ? hi[W1 + t] : S(0));
    }
    S* out = static_cast<S*>(conv_final) + sr * W1;
#pragma unroll
    for (int i = 0; i < 3; ++i)
        if (i < W1) out[i] = v[i];
}

cudaError_t launch_conv_history(const void* x, const void* conv_init, void* conv_final, const int* state_indices,
                                int Bsz, int D, int L, int W1, int dtype, cudaStream_t stream) {
    if (W1 < 1 || W1 > 3) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((D + kConvThreads - 1) / kConvThreads), (unsigned)Bsz);
    if (dtype == 1)
        conv_history_kernel<BF16><<<grid, kConvThreads, 0, stream>>>(x, conv_init, conv_final, state_indices, D, L, W1);
    else
        conv_history_kernel<F32><<<grid, kConvThreads, 0, stream>>>(x, conv_init, conv_final, state_indices, D, L, W1);
    return cudaGetLastError();
}

}  // namespace ssm
