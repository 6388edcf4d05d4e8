// Selective-scan kernels (sequential-in-time, one (b, d) row per thread, fp32 state in registers).
//
// Work decomposition.  A block owns 128 consecutive channels of one batch row and one L segment.
// Each thread walks its channel's segment in time order with all N states in registers, so the
// recurrence h_t = Abar h_{t-1} + Bbar v_t (dpshk.com/news/3333417 sections 2.2/2.3, diagonal A of
// section 3.2) costs no exchange between threads.  B_t and C_t are shared by every channel of a
// batch row (lshu.cn/news/79586 section 3.1), so the block stages them for 64 timesteps at a time
// in shared memory as fp32 and every thread reads them with broadcast loads.
//
// L split.  When B*D rows cannot fill the GPU, L is cut into segments.  A summary pass runs every
// segment but the last from a zero state and records its end state and the sum of its dt (the
// segment's decay is exp(A * sum dt)); the final pass then starts segment s from
//   h_start(s) = exp(A S_{s-1}) h_start(s-1) + hsum_{s-1},   h_start(0) = h0,
// which is the segment state passing of pwwt.cn/news/5168881 section 3.1 done in parallel.
//
// Zero-order hold, per state n with a = A[d, n], x = dt a, Abar = 2^(x log2 e):
//   h' = Abar h + E B v,  E = (exp(x) - 1) / a  (zoh_factor: the Taylor series of expm1(x) / x below
//   |x| = 2^-4, where (Abar - 1) / a would cancel, and the quotient above; dt at a = 0).
#pragma once

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

template <int NS>
struct ScanShared {
    float bc[2][kScanChunk][NS];  // [0] = B_t[n], [1] = C_t[n], fp32, zero past L and past N
};

// Per-thread constants of one channel.
template <int NS>
struct ChannelConsts {
    float al2[NS];   // A[d, n] * log2(e); 0 for padded n >= N
    float inva[NS];  // 1 / A[d, n]; 0 for padded n and for A == 0
    float w[4];      // conv taps aligned so w[3] multiplies x_t
    float cb, dskip, bias;
};

// One group of up to 8 timesteps.  kTail: the group may be partial (nv < 8) or rows unaligned.
template <typename Tin, typename Tout, int NS, Disc kDisc, bool kFinal, bool kTail>
__device__ __forceinline__ void scan_group(const ScanKernelArgs& a, const ScanShared<NS>& sh, int g, size_t rowoff,
                                           int tg, int nv, const ChannelConsts<NS>& cc, float (&h)[NS],
                                           float (&xh)[3], float& dsum, float* hall) {
    float xv[8], dv[8], zv[8];
    const bool has_z = kFinal && a.z != nullptr;
    if (!kTail) {
        load8<Tin>(a.u, rowoff + tg, xv);
        load8<Tin>(a.delta, rowoff + tg, dv);
        if (has_z) load8<Tin>(a.z, rowoff + tg, zv);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            bool ok = j < nv;
            xv[j] = ok ? load1<Tin>(a.u, rowoff + tg + j) : 0.0f;
            dv[j] = ok ? load1<Tin>(a.delta, rowoff + tg + j) : 0.0f;
            zv[j] = (ok && has_z) ? load1<Tin>(a.z, rowoff + tg + j) : 0.0f;
        }
    }

    // Per-timestep scalars: SSM input v (optionally SiLU of the causal conv), step dt, gate.
    float v[8], dt[8], gate[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (a.conv_w != nullptr) {
            float acc = fmaf(cc.w[0], xh[0], cc.cb);
            acc = fmaf(cc.w[1], xh[1], acc);
            acc = fmaf(cc.w[2], xh[2], acc);
            acc = fmaf(cc.w[3], xv[j], acc);
            xh[0] = xh[1];
            xh[1] = xh[2];
            xh[2] = xv[j];
            v[j] = silu(acc);
        } else {
            v[j] = xv[j];
        }
        float s = dv[j] + cc.bias;
        dt[j] = a.softplus ? softplus(s) : s;
        if (kFinal) gate[j] = has_z ? silu(zv[j]) : 1.0f;
    }

    float out[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (kTail && j >= nv) {
            out[j] = 0.0f;
            continue;
        }
        const float* Bt = sh.bc[0][g + j];
        const float* Ct = sh.bc[1][g + j];
        const float dtj = dt[j], vj = v[j];
        float y0 = 0.0f, y1 = 0.0f;
        if (!kFinal) dsum += dtj;
        if (kDisc == Disc::kSimple) {
            const float dv_ = dtj * vj;
#pragma unroll
            for (int n = 0; n < NS; ++n) {
                const float ab = abar_exact(dtj * cc.al2[n]);
                h[n] = fmaf(ab, h[n], dv_ * Bt[n]);
                if (kFinal) {
                    if (n & 1) y1 = fmaf(Ct[n], h[n], y1);
                    else y0 = fmaf(Ct[n], h[n], y0);
                }
            }
        } else {  // zero-order hold, exact form: Bbar = E B with E from zoh_factor (any a, a = 0 included)
#pragma unroll
            for (int n = 0; n < NS; ++n) {
                float ab;
                const float E = zoh_exact(dtj, dtj * cc.al2[n], cc.inva[n], ab);
                h[n] = fmaf(ab, h[n], E * (Bt[n] * vj));
                if (kFinal) {
                    if (n & 1) y1 = fmaf(Ct[n], h[n], y1);
                    else y0 = fmaf(Ct[n], h[n], y0);
                }
            }
        }
        if (kFinal) out[j] = fmaf(cc.dskip, vj, y0 + y1) * gate[j];
        if (kFinal && hall != nullptr && (a.hall_every <= 1 || j == 7 || tg + j == a.L - 1)) {
            // the state after step tg + j: row (b, tg + j, d) of h_all, stride D * N per step; or, after a
            // group's last step (tg is a multiple of 8), row (b, tg / 8, d) of the checkpoints
            float* hp = hall + (size_t)(a.hall_every <= 1 ? tg + j : tg / 8) * a.D * a.N;
            if (a.N == NS && (reinterpret_cast<uintptr_t>(a.h_all) & 15) == 0) {  // whole rows: 16-byte stores
#pragma unroll
                for (int n = 0; n < NS; n += 4)
                    *reinterpret_cast<float4*>(hp + n) = make_float4(h[n], h[n + 1], h[n + 2], h[n + 3]);
            } else {
#pragma unroll
                for (int n = 0; n < NS; ++n)
                    if (n < a.N) hp[n] = h[n];
            }
        }
    }

    if (kFinal) {
        if (!kTail) {
            store8<Tout>(a.y, rowoff + tg, out);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < nv) store1<Tout>(a.y, rowoff + tg + j, out[j]);
        }
    }
}

template <typename Tin, typename Tout, int NS, Disc kDisc, bool kFinal>
__device__ __forceinline__ void scan_segment(const ScanKernelArgs& a, ScanShared<NS>& sh, bool active, int b, size_t row,
                                             int t_begin, int t_end, const ChannelConsts<NS>& cc, float (&h)[NS],
                                             float (&xh)[3], float& dsum, float* hall) {
    const size_t rowoff = row * (size_t)a.L;
    for (int c0 = t_begin; c0 < t_end; c0 += kScanChunk) {
        const int clen = min(kScanChunk, t_end - c0);
        __syncthreads();  // every thread is done reading the previous chunk
        for (int i = threadIdx.x; i < 2 * NS * kScanChunk; i += kScanThreads) {
            const int which = i / (NS * kScanChunk);
            const int rem = i - which * (NS * kScanChunk);
            const int n = rem / kScanChunk;
            const int t = rem - n * kScanChunk;
            float val = 0.0f;
            if (n < a.N && t < clen)
                val = load1<Tin>(which ? a.Cm : a.Bm, ((size_t)b * a.N + n) * a.L + c0 + t);
            sh.bc[which][t][n] = val;
        }
        __syncthreads();
        if (active) {
            for (int g = 0; g < clen; g += 8) {
                const int nv = min(8, clen - g);
                if (a.vec && nv == 8)
                    scan_group<Tin, Tout, NS, kDisc, kFinal, false>(a, sh, g, rowoff, c0 + g, 8, cc, h, xh, dsum, hall);
                else
                    scan_group<Tin, Tout, NS, kDisc, kFinal, true>(a, sh, g, rowoff, c0 + g, nv, cc, h, xh, dsum, hall);
            }
        }
    }
}

// kFinal = false: summary pass over segments 0 .. nseg-2 (grid.z = nseg - 1).
// kFinal = true : output pass over all segments (grid.z = nseg).
template <typename Tin, typename Tout, int NS, bool kZOH, bool kFinal>
__global__ void __launch_bounds__(kScanThreads) scan_seq_kernel(const ScanKernelArgs a) {
    __shared__ ScanShared<NS> sh;
    const int b = blockIdx.y;
    const int seg = blockIdx.z;
    const int d = blockIdx.x * kScanThreads + threadIdx.x;
    const bool active = d < a.D;
    const size_t rows = (size_t)a.Bsz * a.D;
    const size_t row = (size_t)b * a.D + (active ? d : 0);
    const int t_begin = seg * a.seg_len;
    const int t_end = min(a.L, t_begin + a.seg_len);
    // The row's state slot (state_indices: a cache indexed by request; negative = padding row).  h0,
    // h_out and conv_init are indexed by it; u, delta, z, y, B, C by the batch row.
    const int slot = a.state_indices != nullptr ? __ldg(a.state_indices + b) : b;
    const bool pad = slot < 0;
    const size_t srow = (size_t)(pad ? 0 : slot) * a.D + (active ? d : 0);
    const int hsteps = a.hall_every <= 1 ? a.L : (a.L + 7) / 8;  // rows of h_all per batch row
    float* hall = (kFinal && a.h_all != nullptr && active && !pad) ? a.h_all + ((size_t)b * hsteps * a.D + d) * a.N
                                                                  : nullptr;

    ChannelConsts<NS> cc;
#pragma unroll
    for (int n = 0; n < NS; ++n) {
        const float av = (active && n < a.N) ? __ldg(a.A + (size_t)d * a.N + n) : 0.0f;
        cc.al2[n] = av * kLog2e;
        cc.inva[n] = (av != 0.0f) ? 1.0f / av : 0.0f;
    }
    cc.w[0] = cc.w[1] = cc.w[2] = cc.w[3] = 0.0f;
    cc.cb = 0.0f;
    if (a.conv_w != nullptr && active) {
        const int W = a.conv_width;
#pragma unroll
        for (int i = 0; i < 4; ++i)  // tap i of the 4-wide window is tap i - (4 - W) of the filter
            cc.w[i] = i >= 4 - W ? __ldg(a.conv_w + (size_t)d * W + i - (4 - W)) : 0.0f;
        if (a.conv_b != nullptr) cc.cb = __ldg(a.conv_b + d);
    }
    cc.dskip = (a.Dskip != nullptr && active) ? __ldg(a.Dskip + d) : 0.0f;
    cc.bias = (a.delta_bias != nullptr && active) ? __ldg(a.delta_bias + d) : 0.0f;

    // Conv history x_{t-3}, x_{t-2}, x_{t-1} at the segment start: before t = 0 it is the caller's
    // conv_init (the last W - 1 inputs of the previous call, oldest first), else zero.
    float xh[3] = {0.0f, 0.0f, 0.0f};
    if (a.conv_w != nullptr && active) {
        const size_t rowoff = row * (size_t)a.L;
        const int W1 = a.conv_width - 1;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const int t = t_begin - 3 + k;
            if (t >= 0) xh[k] = load1<Tin>(a.u, rowoff + t);
            else if (a.conv_init != nullptr && t >= -W1 && !pad) xh[k] = load1<Tin>(a.conv_init, srow * W1 + W1 + t);
        }
    }

    float h[NS];
    float dsum = 0.0f;
#pragma unroll
    for (int n = 0; n < NS; ++n) h[n] = 0.0f;

    if (kFinal) {
        const float* h0 = (a.nseg > 1) ? a.ws_h0 : a.h0;
        const size_t h0row = (a.nseg > 1) ? row : srow;  // the L split is never planned with state slots
        if (h0 != nullptr && active && !pad) {
#pragma unroll
            for (int n = 0; n < NS; ++n)
                if (n < a.N) h[n] = h0[h0row * a.N + n];
        }
        // Fold in the summaries of the earlier segments.
        for (int s = 0; s < seg; ++s) {
            const float S = active ? a.ws_dsum[(size_t)s * rows + row] : 0.0f;
#pragma unroll
            for (int n = 0; n < NS; ++n) {
                const float hs = (active && n < a.N) ? a.ws_h[((size_t)s * rows + row) * a.N + n] : 0.0f;
                h[n] = fmaf(ex2(cc.al2[n] * S), h[n], hs);
            }
        }
    } else if (seg == 0 && a.ws_h0 != nullptr && a.h0 != nullptr && active) {
        // Copy h0 aside before the final pass may overwrite it through an aliased h_out.
#pragma unroll
        for (int n = 0; n < NS; ++n)
            if (n < a.N) a.ws_h0[row * a.N + n] = a.h0[row * a.N + n];
    }

    // the fp32 path always takes the exact zero-order hold (its bound 1e-4 (1 + |y|) leaves no room for
    // the fast form's error at small |A|)
    constexpr Disc kMain = kZOH ? Disc::kZOHExact : Disc::kSimple;
    const bool run = active && !pad;
    scan_segment<Tin, Tout, NS, kMain, kFinal>(a, sh, run, b, row, t_begin, t_end, cc, h, xh, dsum, hall);

    if (!active) return;
    if (pad) {  // a padding row: y is zero, no slot is touched
        if (kFinal)
            for (int t = t_begin; t < t_end; ++t) store1<Tout>(a.y, row * (size_t)a.L + t, 0.0f);
        return;
    }
    if (kFinal) {
        if (seg == a.nseg - 1 && a.h_out != nullptr) {
            const size_t orow = (a.nseg > 1) ? row : srow;
#pragma unroll
            for (int n = 0; n < NS; ++n)
                if (n < a.N) a.h_out[orow * a.N + n] = h[n];
        }
    } else {
        a.ws_dsum[(size_t)seg * rows + row] = dsum;
#pragma unroll
        for (int n = 0; n < NS; ++n)
            if (n < a.N) a.ws_h[((size_t)seg * rows + row) * a.N + n] = h[n];
    }
}

template <typename Tin, typename Tout, int NS, bool kZOH>
cudaError_t launch_scan_ns(const ScanKernelArgs& a, cudaStream_t stream) {
    dim3 block(kScanThreads);
    const unsigned gx = (unsigned)((a.D + kScanThreads - 1) / kScanThreads);
    if (a.nseg > 1) {
        dim3 grid(gx, (unsigned)a.Bsz, (unsigned)(a.nseg - 1));
        scan_seq_kernel<Tin, Tout, NS, kZOH, false><<<grid, block, 0, stream>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    dim3 grid(gx, (unsigned)a.Bsz, (unsigned)a.nseg);
    scan_seq_kernel<Tin, Tout, NS, kZOH, true><<<grid, block, 0, stream>>>(a);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t launch_scan_typed(const ScanKernelArgs& a, int zoh, cudaStream_t stream) {
    if (a.N <= 4) return zoh ? launch_scan_ns<Tin, Tout, 4, true>(a, stream) : launch_scan_ns<Tin, Tout, 4, false>(a, stream);
    if (a.N <= 8) return zoh ? launch_scan_ns<Tin, Tout, 8, true>(a, stream) : launch_scan_ns<Tin, Tout, 8, false>(a, stream);
    return zoh ? launch_scan_ns<Tin, Tout, 16, true>(a, stream) : launch_scan_ns<Tin, Tout, 16, false>(a, stream);
}

}  // namespace ssm
