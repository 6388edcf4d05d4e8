// Backward pass of the selective scan (training; pwwt.cn/news/5168881 section 3.2: the gradient runs
// back along time through the state recurrence).  One thread per (b, d) row, all N states and their
// adjoints in registers, walking time in reverse:
//
//   forward (per step t, state n):  x = dt a,  Abar = e^x,  E = (Abar - 1) / a  (ZOH; dt when a = 0)
//                                   or E = dt (simplified),  h_t = Abar h_{t-1} + E B v,
//                                   y_t = (sum_n C h_t + D v) SiLU(z)
//   backward:  g_n (adjoint of h_t) += C dyss;  dC += dyss h_t;  dAbar = g h_{t-1};  dBbar = g v;
//              dv += g E B;  dB += dBbar E;  dE = dBbar B;
//              d(dt) += dAbar Abar a + dE dE/d(dt);  da += dAbar Abar dt + dE dE/da;  g <- Abar g
//   with dE/d(dt) = Abar, dE/da = (dt Abar - E) / a (dt^2 / 2 at a = 0) for ZOH; 1 and 0 simplified.
//   E and dE/da come from zoh_factor2 / zoh_factor_da2 (packed pairs): Taylor series where |x| is small,
//   so that neither cancels as x -> 0.
//
// The states h_t are recomputed from the forward call's checkpoints (h_ckpt: the state after every 8th
// step, (B, ceil(L/8), D, N); the gradient checkpointing of pwwt.cn/news/5168881 section 3.2 in place of
// keeping every state): before each group of 8 steps, thread (b, d) reloads the checkpoint that precedes
// it (64 contiguous bytes) and runs the group's recurrence forward again, keeping the 8 states in shared
// memory, then walks them in reverse.  Everything else (conv front end, dt, Abar, E) is recomputed from
// the inputs.  dB and dC are sums over the channels of a batch
// row: per step each warp transposes its lanes' contributions through shared memory and sums them, and
// after a group of 8 steps the block adds its four warp sums to global memory with one atomic per (b, n,
// t).  Per-channel parameter gradients (dA, D skip, dt bias, conv taps and bias) accumulate over time in
// registers and are added atomically over the batch at the end; the host zeroes them first.
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

namespace {

constexpr int kBwdThreads = 128;
constexpr int kBwdChunk = 64;   // steps of B / C staged per chunk
constexpr int kBwdGroup = 8;    // steps per group (vector loads / stores, one reduction flush)
constexpr int kCkpt = SSM_CKPT_STEPS;  // steps per forward checkpoint: one group
static_assert(kCkpt == kBwdGroup, "a group starts right after a checkpoint");

// Per-thread scalars of a group kept in shared memory for the reverse walk (a step loop that is not
// unrolled would otherwise index register arrays at run time, which puts them in local memory, and with
// two blocks' shared memory on the SM the L1 left over cannot hold that): per step dt, the softplus
// argument s, the conv output c (the SSM input v without conv) and dy, z; then x_{tg-3} .. x_{tg+7}.
enum BwdField { kFDt = 0, kFS, kFC, kFGy, kFZ, kFX };
constexpr int kBwdScalars = kFX * kBwdGroup + kBwdGroup + 3;

// Dynamic shared memory of the backward kernel: the group's recomputed states h_tg .. h_tg+6 (h_tg+7
// stays in registers), then the scalars above.
template <int NS>
constexpr int bwd_state_smem() {
    return ((kBwdGroup - 1) * NS + kBwdScalars) * kBwdThreads * (int)sizeof(float);
}

template <int NS>
struct BwdShared {
    float bc[2][kBwdChunk][NS];               // B_t[n], C_t[n] of the chunk, fp32
    float tr[kBwdThreads / 32][32][36];       // per warp: a row of 32 values per lane (padded to 36)
    float ws[kBwdThreads / 32][kBwdGroup][32];  // per-warp sums of the group's steps
};

__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + ex2(-x * kLog2e)); }

template <typename T>
__device__ __forceinline__ float ld(const void* p, size_t i, bool ok) {
    return ok ? load1<T>(p, i) : 0.0f;
}

// zoh_factor2 given 1/a instead of -1/a ((Abar - 1)(1/a) is (1 - Abar)(-1/a) exactly): the kernel keeps one
// reciprocal per state in registers, not two.
__device__ __forceinline__ f32x2 zoh_e2(f32x2 dt2, f32x2 y2, f32x2 ab2, f32x2 inva2) {
    f32x2 p = fma2(y2, pack2(kPhiY3, kPhiY3), pack2(kPhiY2, kPhiY2));
    p = fma2(p, y2, pack2(kPhiY1, kPhiY1));
    p = fma2(p, y2, pack2(1.0f, 1.0f));
    const f32x2 small = mul2(p, dt2);
    const f32x2 big = mul2(sub2(ab2, pack2(1.0f, 1.0f)), inva2);
    float y0, y1, s0, s1, b0, b1;
    unpack2(y2, y0, y1);
    unpack2(small, s0, s1);
    unpack2(big, b0, b1);
    return pack2(fabsf(y0) < kZohSeriesY ? s0 : b0, fabsf(y1) < kZohSeriesY ? s1 : b1);
}

// Asks L2 for the line that holds element i of base; no register waits on it.
template <typename T>
__device__ __forceinline__ void prefetch_l2(const void* base, size_t i) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char*>(base) + i * T::kBytes));
}

template <typename Tin, int NS, bool kZOH, bool kConv>
__global__ void __launch_bounds__(kBwdThreads) scan_bwd_kernel(const ScanBwdArgs a) {
    __shared__ BwdShared<NS> sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.y, seg = blockIdx.z;
    const int d = blockIdx.x * kBwdThreads + tid;
    const bool active = d < a.D;
    const int dd = active ? d : 0;
    const size_t row = (size_t)b * a.D + dd;
    const size_t rowoff = row * (size_t)a.L;
    const int L = a.L, N = a.N;
    const size_t rows = (size_t)a.Bsz * a.D;
    const int t0 = seg * a.seg_len;                // this block's steps: [t0, t1)
    const int t1 = min(L, t0 + a.seg_len);

    // per-channel constants, as packed pairs of states (n, n + 1)
    // (the exponent argument dt a log2 e is formed as (dt log2 e) a, one scalar product per step)
    f32x2 a2[NS / 2], inva2[NS / 2];
    bool small_a = false;   // some state of this channel with |A| < kZohFastMinA (0 included)
#pragma unroll
    for (int p = 0; p < NS / 2; ++p) {
        float av[2], iv[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int n = 2 * p + q;
            const bool real = active && n < N;
            av[q] = real ? __ldg(a.A + (size_t)dd * N + n) : 0.0f;
            iv[q] = av[q] != 0.0f ? 1.0f / av[q] : 0.0f;
            small_a |= real && !(fabsf(av[q]) >= kZohFastMinA);
        }
        a2[p] = pack2(av[0], av[1]);
        inva2[p] = pack2(iv[0], iv[1]);
    }
    // Block-uniform: with bf16 inputs and every |A| of the block at least kZohFastMinA, the forward pass
    // took the fast form h' = Abar (h - ng) + ng, ng = -(v / a) B; the recomputation of a group's states
    // takes it too (fewer products than the exact E, and the same rounding as the forward's states).
    const bool fast_rc = kZOH && Tin::kBytes == 2 && !__syncthreads_or(small_a);
    float w[4] = {0.0f, 0.0f, 0.0f, 0.0f}, cb = 0.0f;
    if (kConv && active) {
        const int W = a.conv_width;
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = i >= 4 - W ? __ldg(a.conv_w + (size_t)dd * W + i - (4 - W)) : 0.0f;
        if (a.conv_b) cb = __ldg(a.conv_b + dd);
    }
    const float dsk = (a.Dskip && active) ? __ldg(a.Dskip + dd) : 0.0f;
    const float bias = (a.delta_bias && active) ? __ldg(a.delta_bias + dd) : 0.0f;
    const bool has_z = a.z != nullptr;

    // adjoint of the state at the segment's end: dh_out carried back through the later segments with
    // their summaries, g <- exp(a sum dt) g + g_local in reverse segment order; and the accumulators
    f32x2 g2[NS / 2], da2[NS / 2];
#pragma unroll
    for (int p = 0; p < NS / 2; ++p) {
        float gv[2];
#pragma unroll
        for (int q = 0; q < 2; ++q)
            gv[q] = (a.dh_out && active && 2 * p + q < N) ? a.dh_out[row * N + 2 * p + q] : 0.0f;
        g2[p] = pack2(gv[0], gv[1]);
        da2[p] = pack2(0.0f, 0.0f);
    }
    for (int s2 = a.nseg - 1; s2 > seg; --s2) {
        const float S = active ? a.ws_dsum[(size_t)(s2 - 1) * rows + row] : 0.0f;
        const float* gl = a.ws_g + ((size_t)(s2 - 1) * rows + row) * N;
#pragma unroll
        for (int p = 0; p < NS / 2; ++p) {
            float gv[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) gv[q] = (active && 2 * p + q < N) ? gl[2 * p + q] : 0.0f;
            g2[p] = fma2(ex2x2(mul2(pack2(S * kLog2e, S * kLog2e), a2[p])), g2[p], pack2(gv[0], gv[1]));
        }
    }
    float dD = 0.0f, dbias = 0.0f, dw[4] = {0.0f, 0.0f, 0.0f, 0.0f}, dcb = 0.0f;
    float px[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // pending dx of x_t, x_{t-1}, x_{t-2}, x_{t-3}

    // The group's states h_tg .. h_tg+7, recomputed from the checkpoint before the group, live in
    // dynamic shared memory as [step j][quad q][thread] float4s (conflict-free 16-byte accesses); the
    // state before the group, h_{tg-1}, stays in registers.
    extern __shared__ float4 bwd_hs[];
    auto hs_at = [&](int j, int q) -> float4& { return bwd_hs[(j * (NS / 4) + q) * kBwdThreads + tid]; };
    float* const bwd_sc = reinterpret_cast<float*>(bwd_hs + (kBwdGroup - 1) * (NS / 4) * kBwdThreads);
    auto sc_at = [&](int f, int j) -> float& { return bwd_sc[(f * kBwdGroup + j) * kBwdThreads + tid]; };
    const int nck = (L + kCkpt - 1) / kCkpt;
    const float* crow = a.h_ckpt + ((size_t)b * nck * a.D + dd) * N;  // entry c: the state after step 8c + 7
    const size_t cstride = (size_t)a.D * N;

    const int last_chunk = t0 + ((t1 - 1 - t0) / kBwdChunk) * kBwdChunk;
    for (int c0 = last_chunk; c0 >= t0; c0 -= kBwdChunk) {
        const int clen = min(kBwdChunk, t1 - c0);
        __syncthreads();  // everyone is done with the previous chunk's B / C
        {
            // all of a thread's loads first, then the stores (one memory latency per chunk)
            constexpr int kStage = 2 * NS * kBwdChunk / kBwdThreads;
            float stage[kStage];
#pragma unroll
            for (int r = 0; r < kStage; ++r) {
                const int i = tid + r * kBwdThreads;
                const int wv = i / (NS * kBwdChunk);
                const int rem = i - wv * NS * kBwdChunk;
                const int n = rem / kBwdChunk, t = rem - n * kBwdChunk;
                stage[r] = (n < N && t < clen) ? load1<Tin>(wv ? a.Cm : a.Bm, ((size_t)b * N + n) * L + c0 + t) : 0.0f;
            }
#pragma unroll
            for (int r = 0; r < kStage; ++r) {
                const int i = tid + r * kBwdThreads;
                const int wv = i / (NS * kBwdChunk);
                const int rem = i - wv * NS * kBwdChunk;
                const int n = rem / kBwdChunk, t = rem - n * kBwdChunk;
                sh.bc[wv][t][n] = stage[r];
            }
        }
        // the next chunk's B / C rows into L2 while this chunk runs
        if (c0 - kBwdChunk >= t0 && tid < 2 * NS && tid % NS < N) {
            const void* base = tid >= NS ? a.Cm : a.Bm;
            const size_t o = ((size_t)b * N + tid % NS) * L + c0 - kBwdChunk;
            prefetch_l2<Tin>(base, o);
            prefetch_l2<Tin>(base, o + kBwdChunk / 2);
            prefetch_l2<Tin>(base, o + kBwdChunk - 1);
        }
        __syncthreads();
        const int last_group = ((clen - 1) / kBwdGroup) * kBwdGroup;
        for (int g0 = last_group; g0 >= 0; g0 -= kBwdGroup) {
            const int tg = c0 + g0;
            const int nv = min(kBwdGroup, clen - g0);
            // inputs of the group's steps, and the conv inputs x_{tg-3} .. x_{tg-1} before them
            float xv[kBwdGroup], dv[kBwdGroup], zv[kBwdGroup], gy[kBwdGroup], xh[3];
            if (a.vec && nv == kBwdGroup && active) {  // 16-byte rows: vector loads
                load8<Tin>(a.u, rowoff + tg, xv);
                load8<Tin>(a.delta, rowoff + tg, dv);
                if (has_z) load8<Tin>(a.z, rowoff + tg, zv);
                load8<Tin>(a.dy, rowoff + tg, gy);
                if (!has_z) {
#pragma unroll
                    for (int j = 0; j < kBwdGroup; ++j) zv[j] = 0.0f;
                }
            } else {
#pragma unroll
                for (int j = 0; j < kBwdGroup; ++j) {
                    const bool ok = active && j < nv;
                    xv[j] = ld<Tin>(a.u, rowoff + tg + j, ok);
                    dv[j] = ld<Tin>(a.delta, rowoff + tg + j, ok);
                    zv[j] = has_z ? ld<Tin>(a.z, rowoff + tg + j, ok) : 0.0f;
                    gy[j] = ld<Tin>(a.dy, rowoff + tg + j, ok);
                }
            }
            // the state before the group (the previous group's checkpoint, or h0), loaded with the inputs so
            // that the two latencies overlap
            f32x2 hstart[NS / 2];
            {
                const float* src = tg > 0 ? crow + (size_t)(tg / kCkpt - 1) * cstride : a.h0 ? a.h0 + row * N : nullptr;
                // src is NULL before t = 0 without h0: the state is zero, nothing is read
                const bool vec4 = src != nullptr && (N == NS) && ((reinterpret_cast<uintptr_t>(src) & 15) == 0);
                if (vec4 && active) {
                    const ulonglong2* q = reinterpret_cast<const ulonglong2*>(src);
#pragma unroll
                    for (int k = 0; k < NS / 4; ++k) {
                        const ulonglong2 w2 = __ldcs(q + k);
                        hstart[2 * k] = w2.x;
                        hstart[2 * k + 1] = w2.y;
                    }
                } else {
#pragma unroll
                    for (int p = 0; p < NS / 2; ++p) {
                        float hv[2];
#pragma unroll
                        for (int q = 0; q < 2; ++q) hv[q] = (src && active && 2 * p + q < N) ? src[2 * p + q] : 0.0f;
                        hstart[p] = pack2(hv[0], hv[1]);
                    }
                }
            }
            // the next group's rows (the eight steps before this one) and its checkpoint into L2 while
            // this group runs
            if (active && tg - kBwdGroup >= t0) {
                const size_t o = rowoff + tg - kBwdGroup;
                prefetch_l2<Tin>(a.u, o);
                prefetch_l2<Tin>(a.delta, o);
                if (has_z) prefetch_l2<Tin>(a.z, o);
                prefetch_l2<Tin>(a.dy, o);
                if (tg - kBwdGroup > 0) prefetch_l2<F32>(crow, (size_t)((tg - kBwdGroup) / kCkpt - 1) * cstride);
            }
            if (kConv) {
                const int W1 = a.conv_width - 1;
#pragma unroll
                for (int k = 0; k < 3; ++k) {
                    const int t = tg - 3 + k;
                    xh[k] = 0.0f;
                    if (active && t >= 0) xh[k] = load1<Tin>(a.u, rowoff + t);
                    else if (active && a.conv_init && t >= -W1) xh[k] = load1<Tin>(a.conv_init, row * W1 + W1 + t);
                }
            }
            // per-step scalars of the group: SSM input v (conv output c), step dt; kept for the reverse walk
            float vv[kBwdGroup], dtv[kBwdGroup];
#pragma unroll
            for (int j = 0; j < kBwdGroup; ++j) {
                float v;
                if (kConv) {
                    float xm[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int m = j - 3 + k;  // x_{t-3+k}
                        xm[k] = m >= 0 ? xv[m >= 0 ? m : 0] : xh[m + 3 >= 0 ? m + 3 : 0];
                    }
                    float c = fmaf(w[0], xm[0], cb);
                    c = fmaf(w[1], xm[1], c);
                    c = fmaf(w[2], xm[2], c);
                    c = fmaf(w[3], xm[3], c);
                    v = c * sigmoid_f(c);  // SiLU, formed as the reverse walk forms it
                    sc_at(kFC, j) = c;
                } else {
                    v = xv[j];
                    sc_at(kFC, j) = v;
                }
                vv[j] = v;
                const float sj = dv[j] + bias;
                dtv[j] = a.softplus ? softplus(sj) : sj;
                sc_at(kFDt, j) = dtv[j];
                sc_at(kFS, j) = sj;
                sc_at(kFGy, j) = gy[j];
                sc_at(kFZ, j) = zv[j];
            }
            if (kConv) {
#pragma unroll
                for (int k = 0; k < 3; ++k) sc_at(kFX, k) = xh[k];
#pragma unroll
                for (int j = 0; j < kBwdGroup; ++j) sc_at(kFX, 3 + j) = xv[j];
            }
            // the group's states recomputed forward from the state before it with the forward pass's
            // zero-order hold (exact form)
            f32x2 hcur[NS / 2];
            {
#pragma unroll
                for (int p = 0; p < NS / 2; ++p) hcur[p] = hstart[p];
#pragma unroll
                for (int j = 0; j < kBwdGroup; ++j) {
                    if (j >= nv) break;  // uniform over the block
                    const f32x2* Bt = reinterpret_cast<const f32x2*>(sh.bc[0][tg + j - c0]);
                    const f32x2 dt2 = pack2(dtv[j], dtv[j]), v2 = pack2(vv[j], vv[j]);
                    const float dtl = dtv[j] * kLog2e;
                    const f32x2 dtl2 = pack2(dtl, dtl);
                    if (fast_rc) {
#pragma unroll
                        for (int p = 0; p < NS / 2; ++p) {
                            const f32x2 Ab = ex2x2(mul2(dtl2, a2[p]));
                            const f32x2 q = mul2(mul2(v2, inva2[p]), Bt[p]);   // -ng = (v / a) B
                            hcur[p] = fma2(Ab, add2(hcur[p], q), mul2(q, pack2(-1.0f, -1.0f)));
                        }
                    } else {
#pragma unroll
                        for (int p = 0; p < NS / 2; ++p) {
                            const f32x2 y2 = mul2(dtl2, a2[p]);
                            const f32x2 Ab = ex2x2(y2);
                            f32x2 E = dt2;
                            if (kZOH) E = zoh_e2(dt2, y2, Ab, inva2[p]);
                            hcur[p] = fma2(Ab, hcur[p], mul2(E, mul2(v2, Bt[p])));
                        }
                    }
                    if (j == kBwdGroup - 1) break;  // the group's last state stays in hcur
#pragma unroll
                    for (int k = 0; k < NS / 4; ++k) {
                        float h0_, h1_, h2_, h3_;
                        unpack2(hcur[2 * k], h0_, h1_);
                        unpack2(hcur[2 * k + 1], h2_, h3_);
                        hs_at(j, k) = make_float4(h0_, h1_, h2_, h3_);
                    }
                }
            }
            // not unrolled: the step body is large (eight state pairs), and eight copies of it overflow the
            // instruction cache (4.86 -> 4.48 ms on the 8 x 4096 x 16 x 2048 layer); the per-step scalars
            // come from shared memory, and the step's input gradients go back into its dt, s and z slots
#pragma unroll 1
            for (int j = kBwdGroup - 1; j >= 0; --j) {
                if (j >= nv) continue;  // uniform over the block: nv is
                const int t = tg + j;
                const float dt = sc_at(kFDt, j), s = sc_at(kFS, j), gyj = sc_at(kFGy, j), zj = sc_at(kFZ, j);
                float c = 0.0f, sgc = 0.0f, v;
                if (kConv) {
                    c = sc_at(kFC, j);
                    sgc = sigmoid_f(c);
                    v = c * sgc;
                } else {
                    v = sc_at(kFC, j);
                }
                float xm[4];
                if (kConv) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) xm[k] = sc_at(kFX, j + k);  // x_{t-3+k}
                }
                // h_t (in hcur since the previous step, or from the forward recompute) and h_{t-1}
                f32x2 hprev[NS / 2];
                if (j > 0) {
#pragma unroll
                    for (int k = 0; k < NS / 4; ++k) {
                        const float4 f = hs_at(j - 1, k);
                        hprev[2 * k] = pack2(f.x, f.y);
                        hprev[2 * k + 1] = pack2(f.z, f.w);
                    }
                } else {
#pragma unroll
                    for (int p = 0; p < NS / 2; ++p) hprev[p] = hstart[p];
                }
                const f32x2* Bt = reinterpret_cast<const f32x2*>(sh.bc[0][t - c0]);
                const f32x2* Ct = reinterpret_cast<const f32x2*>(sh.bc[1][t - c0]);
                f32x2 yacc = pack2(0.0f, 0.0f);
#pragma unroll
                for (int p = 0; p < NS / 2; ++p) yacc = fma2(Ct[p], hcur[p], yacc);
                float ya, yb;
                unpack2(yacc, ya, yb);
                const float yss = fmaf(dsk, v, ya + yb);
                float dyss = gyj;
                if (has_z) {
                    const float sg = sigmoid_f(zj);
                    const float gz = zj * sg;
                    sc_at(kFZ, j) = gyj * yss * sg * (1.0f + zj * (1.0f - sg));  // dz
                    dyss = gyj * gz;
                }
                dD = fmaf(dyss, v, dD);
                const f32x2 dyss2 = pack2(dyss, dyss), dt2 = pack2(dt, dt), v2 = pack2(v, v);
                const f32x2 one2 = pack2(1.0f, 1.0f);
                const f32x2 dtsq2 = pack2(dt * dt, dt * dt);
                const float dtl = dt * kLog2e;
                const f32x2 dtl2 = pack2(dtl, dtl);
                f32x2 dvp = pack2(0.0f, 0.0f), ddtp = pack2(0.0f, 0.0f);
                f32x2 red2[16];
#pragma unroll
                for (int p = 0; p < NS / 2; ++p) {
                    g2[p] = fma2(Ct[p], dyss2, g2[p]);
                    red2[8 + p] = mul2(dyss2, hcur[p]);                 // dC contribution
                    const f32x2 y2 = mul2(dtl2, a2[p]);
                    const f32x2 Ab = ex2x2(y2);
                    f32x2 E, dEdt, dEda;
                    if (!kZOH) {
                        E = dt2;
                        dEdt = one2;
                        dEda = pack2(0.0f, 0.0f);
                    } else {
                        // exact forms (zoh_factor2, zoh_factor_da2): Taylor series where |dt a| is small, where
                        // (Abar - 1) / a and (dt Abar - E) / a would cancel; the limits dt and dt^2 / 2 at a = 0
                        E = zoh_e2(dt2, y2, Ab, inva2[p]);
                        dEdt = Ab;
                        dEda = zoh_factor_da2(dt2, dtsq2, mul2(dt2, a2[p]), Ab, E, inva2[p]);
                    }
                    const f32x2 dAb = mul2(g2[p], hprev[p]);
                    const f32x2 dBb = mul2(g2[p], v2);
                    dvp = fma2(mul2(g2[p], E), Bt[p], dvp);
                    red2[p] = mul2(dBb, E);                              // dB contribution
                    const f32x2 dE = mul2(dBb, Bt[p]);
                    const f32x2 tA = mul2(dAb, Ab);
                    ddtp = fma2(tA, a2[p], fma2(dE, dEdt, ddtp));
                    da2[p] = fma2(tA, dt2, fma2(dE, dEda, da2[p]));
                    g2[p] = mul2(g2[p], Ab);
                    hcur[p] = hprev[p];
                }
#pragma unroll
                for (int p = NS / 2; p < 8; ++p) red2[p] = red2[8 + p] = pack2(0.0f, 0.0f);
                float d0, d1;
                unpack2(dvp, d0, d1);
                const float dvv = fmaf(dsk, dyss, d0 + d1);
                unpack2(ddtp, d0, d1);
                const float ddt = d0 + d1;
                const float ds = a.softplus ? ddt * sigmoid_f(s) : ddt;
                dbias += ds;
                sc_at(kFS, j) = ds;  // d delta
                if (kConv) {
                    const float dc = dvv * sgc * (1.0f + c * (1.0f - sgc));
                    dcb += dc;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        dw[k] = fmaf(dc, xm[k], dw[k]);
                        px[3 - k] = fmaf(dc, w[k], px[3 - k]);     // x_{t-3+k} is pending slot 3 - k
                    }
                    sc_at(kFDt, j) = px[0];  // du
                    px[0] = px[1];
                    px[1] = px[2];
                    px[2] = px[3];
                    px[3] = 0.0f;
                } else {
                    sc_at(kFDt, j) = dvv;  // du
                }
                // the warp's sum of each of the 32 values (dB n, dC n): every lane writes its row of 32
                // with 16-byte stores, every lane then sums one column (rows padded to 36 floats: both
                // passes are free of bank conflicts)
                if (!active) {
#pragma unroll
                    for (int k = 0; k < 16; ++k) red2[k] = pack2(0.0f, 0.0f);
                }
                ulonglong2* trow = reinterpret_cast<ulonglong2*>(&sh.tr[warp][lane][0]);
#pragma unroll
                for (int k = 0; k < 8; ++k) trow[k] = make_ulonglong2(red2[2 * k], red2[2 * k + 1]);
                __syncwarp();
                // four independent partial sums: a 32-long chain of dependent adds would cost ~128 cycles
                float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int k = 0; k < 32; ++k) s4[k & 3] += sh.tr[warp][k][lane];
                sh.ws[warp][j][lane] = (s4[0] + s4[1]) + (s4[2] + s4[3]);
                __syncwarp();
            }
            // outputs of the group
            float du_o[kBwdGroup], dd_o[kBwdGroup], dz_o[kBwdGroup];
#pragma unroll
            for (int j = 0; j < kBwdGroup; ++j) {
                du_o[j] = sc_at(kFDt, j);
                dd_o[j] = sc_at(kFS, j);
                dz_o[j] = sc_at(kFZ, j);
            }
            if (active && a.vec && nv == kBwdGroup) {
                store8<Tin>(a.du, rowoff + tg, du_o);
                store8<Tin>(a.ddelta, rowoff + tg, dd_o);
                if (has_z) store8<Tin>(a.dz, rowoff + tg, dz_o);
            } else if (active) {
#pragma unroll
                for (int j = 0; j < kBwdGroup; ++j) {
                    if (j < nv) {
                        store1<Tin>(a.du, rowoff + tg + j, du_o[j]);
                        store1<Tin>(a.ddelta, rowoff + tg + j, dd_o[j]);
                        if (has_z) store1<Tin>(a.dz, rowoff + tg + j, dz_o[j]);
                    }
                }
            }
            // dB, dC of the group: the four warps' sums, one atomic per (n, t)
            __syncthreads();
            for (int i = tid; i < kBwdGroup * 32; i += kBwdThreads) {
                const int j = i >> 5, k = i & 31;
                const int n = k & 15;
                if (j < nv && n < N) {
                    float tot = 0.0f;
#pragma unroll
                    for (int wv = 0; wv < kBwdThreads / 32; ++wv) tot += sh.ws[wv][j][k];
                    float* dst = (k < 16 ? a.dB : a.dC) + ((size_t)b * N + n) * L + tg + j;
                    atomicAdd(dst, tot);
                }
            }
            __syncthreads();
        }
    }

    if (!active) return;
    // the adjoint before t = 0, and the conv history's gradient
    float gl[NS], dal[NS];
#pragma unroll
    for (int p = 0; p < NS / 2; ++p) {
        unpack2(g2[p], gl[2 * p], gl[2 * p + 1]);
        unpack2(da2[p], dal[2 * p], dal[2 * p + 1]);
    }
    if (a.dh0 && seg == 0) {
#pragma unroll
        for (int n = 0; n < NS; ++n)
            if (n < N) a.dh0[row * N + n] = gl[n];
    }
    if (kConv && seg == 0 && a.dconv_init) {
        const int W1 = a.conv_width - 1;
#pragma unroll
        for (int k = 0; k < 3; ++k)  // px[k] holds dx of x_{-1-k}
            if (k < W1) store1<Tin>(a.dconv_init, row * W1 + W1 - 1 - k, px[k]);
    }
    if (kConv && seg > 0) {
        // the input gradients this segment owes to x_{t0-1}, x_{t0-2}, x_{t0-3} (the previous segment's
        // steps): added to du by the boundary pass after every segment is done
        float* pend = a.ws_pend + ((size_t)(seg - 1) * rows + row) * 3;
#pragma unroll
        for (int k = 0; k < 3; ++k) pend[k] = px[k];
    }
#pragma unroll
    for (int n = 0; n < NS; ++n)
        if (n < N) atomicAdd(a.dA + (size_t)dd * N + n, dal[n]);
    if (a.dDskip) atomicAdd(a.dDskip + dd, dD);
    if (a.ddelta_bias) atomicAdd(a.ddelta_bias + dd, dbias);
    if (kConv) {
        const int W = a.conv_width;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (i >= 4 - W && a.dconv_w) atomicAdd(a.dconv_w + (size_t)dd * W + i - (4 - W), dw[i]);
        if (a.dconv_b) atomicAdd(a.dconv_b + dd, dcb);
    }
}

// Summary of segment s >= 1 for the L split: the adjoint it hands to segment s - 1 when it starts from
// zero (g <- g + C_t dyss_t, then g <- Abar_t g, back over the segment), and the segment's sum of dt
// (its decay is exp(a sum dt)).  Needs only dy, z, delta and C: dyss = dy SiLU(z) does not depend on
// the states.  The final pass folds these in reverse segment order.
template <typename Tin, int NS>
__global__ void __launch_bounds__(kBwdThreads) scan_bwd_summary_kernel(const ScanBwdArgs a) {
    __shared__ float cs[kBwdChunk][NS];
    const int tid = threadIdx.x, b = blockIdx.y, seg = blockIdx.z + 1;
    const int d = blockIdx.x * kBwdThreads + tid;
    const bool active = d < a.D;
    const int dd = active ? d : 0;
    const int L = a.L, N = a.N;
    const size_t rows = (size_t)a.Bsz * a.D, row = (size_t)b * a.D + dd, rowoff = row * (size_t)L;
    const int t0 = seg * a.seg_len, t1 = min(L, t0 + a.seg_len);
    f32x2 al2[NS / 2], g2[NS / 2];
#pragma unroll
    for (int p = 0; p < NS / 2; ++p) {
        float av[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) av[q] = (active && 2 * p + q < N) ? __ldg(a.A + (size_t)dd * N + 2 * p + q) : 0.0f;
        al2[p] = pack2(av[0] * kLog2e, av[1] * kLog2e);
        g2[p] = pack2(0.0f, 0.0f);
    }
    const float bias = (a.delta_bias && active) ? __ldg(a.delta_bias + dd) : 0.0f;
    float dsum = 0.0f;
    const int last_chunk = t0 + ((t1 - 1 - t0) / kBwdChunk) * kBwdChunk;
    for (int c0 = last_chunk; c0 >= t0; c0 -= kBwdChunk) {
        const int clen = min(kBwdChunk, t1 - c0);
        __syncthreads();
        for (int i = tid; i < NS * kBwdChunk; i += kBwdThreads) {
            const int n = i / kBwdChunk, t = i - n * kBwdChunk;
            cs[t][n] = (n < N && t < clen) ? load1<Tin>(a.Cm, ((size_t)b * N + n) * L + c0 + t) : 0.0f;
        }
        __syncthreads();
        for (int g0 = ((clen - 1) / kBwdGroup) * kBwdGroup; g0 >= 0; g0 -= kBwdGroup) {
            const int tg = c0 + g0, nv = min(kBwdGroup, clen - g0);
            float dv[kBwdGroup], zv[kBwdGroup], gy[kBwdGroup];
#pragma unroll
            for (int j = 0; j < kBwdGroup; ++j) {
                const bool ok = active && j < nv;
                dv[j] = ld<Tin>(a.delta, rowoff + tg + j, ok);
                zv[j] = a.z ? ld<Tin>(a.z, rowoff + tg + j, ok) : 0.0f;
                gy[j] = ld<Tin>(a.dy, rowoff + tg + j, ok);
            }
#pragma unroll
            for (int j = kBwdGroup - 1; j >= 0; --j) {
                if (j >= nv) continue;
                const float sv = dv[j] + bias;
                const float dt = a.softplus ? softplus(sv) : sv;
                const float dyss = a.z ? gy[j] * zv[j] * sigmoid_f(zv[j]) : gy[j];
                const f32x2 dyss2 = pack2(dyss, dyss), dt2 = pack2(dt, dt);
                const f32x2* Ct = reinterpret_cast<const f32x2*>(cs[tg + j - c0]);
#pragma unroll
                for (int p = 0; p < NS / 2; ++p)
                    g2[p] = mul2(ex2x2(mul2(dt2, al2[p])), fma2(Ct[p], dyss2, g2[p]));
                dsum += dt;
            }
        }
    }
    if (!active) return;
    a.ws_dsum[(size_t)(seg - 1) * rows + row] = dsum;
    float* gl = a.ws_g + ((size_t)(seg - 1) * rows + row) * N;
#pragma unroll
    for (int p = 0; p < NS / 2; ++p) {
        float g0_, g1_;
        unpack2(g2[p], g0_, g1_);
        if (2 * p < N) gl[2 * p] = g0_;
        if (2 * p + 1 < N) gl[2 * p + 1] = g1_;
    }
}

// After the L-split backward: the input gradients each segment s >= 1 owes to the three steps before it
// (conv taps reaching back over the boundary), added to du there.
template <typename Tin>
__global__ void __launch_bounds__(kBwdThreads) scan_bwd_boundary_kernel(const ScanBwdArgs a) {
    const int d = blockIdx.x * kBwdThreads + threadIdx.x, b = blockIdx.y, seg = blockIdx.z + 1;
    if (d >= a.D) return;
    const size_t rows = (size_t)a.Bsz * a.D, row = (size_t)b * a.D + d;
    const float* pend = a.ws_pend + ((size_t)(seg - 1) * rows + row) * 3;
    const int t0 = seg * a.seg_len;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const int t = t0 - 1 - k;
        if (t >= 0) {
            const size_t i = row * (size_t)a.L + t;
            store1<Tin>(a.du, i, load1<Tin>(a.du, i) + pend[k]);
        }
    }
}

template <typename Tin, int NS, bool kZOH>
cudaError_t launch_bwd_z(const ScanBwdArgs& a, cudaStream_t s) {
    const unsigned gx = (unsigned)((a.D + kBwdThreads - 1) / kBwdThreads);
    if (a.nseg > 1) {
        scan_bwd_summary_kernel<Tin, NS><<<dim3(gx, (unsigned)a.Bsz, (unsigned)(a.nseg - 1)), kBwdThreads, 0, s>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    dim3 grid(gx, (unsigned)a.Bsz, (unsigned)a.nseg);
    auto kfn = a.conv_w ? scan_bwd_kernel<Tin, NS, kZOH, true> : scan_bwd_kernel<Tin, NS, kZOH, false>;
    cudaError_t e = set_dynamic_smem_once(kfn, bwd_state_smem<NS>());
    if (e != cudaSuccess) return e;
    kfn<<<grid, kBwdThreads, bwd_state_smem<NS>(), s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess || a.nseg <= 1 || !a.conv_w) return e;
    scan_bwd_boundary_kernel<Tin><<<dim3(gx, (unsigned)a.Bsz, (unsigned)(a.nseg - 1)), kBwdThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin, int NS>
cudaError_t launch_bwd_n(const ScanBwdArgs& a, int zoh, cudaStream_t s) {
    return zoh ? launch_bwd_z<Tin, NS, true>(a, s) : launch_bwd_z<Tin, NS, false>(a, s);
}

template <typename Tin>
cudaError_t launch_bwd_t(const ScanBwdArgs& a, int zoh, cudaStream_t s) {
    if (a.N <= 4) return launch_bwd_n<Tin, 4>(a, zoh, s);
    if (a.N <= 8) return launch_bwd_n<Tin, 8>(a, zoh, s);
    return launch_bwd_n<Tin, 16>(a, zoh, s);
}

template <typename Tin, int NS>
const void* bwd_kernel_ptr(int zoh, bool conv) {
    if (zoh) return conv ? reinterpret_cast<const void*>(scan_bwd_kernel<Tin, NS, true, true>)
                         : reinterpret_cast<const void*>(scan_bwd_kernel<Tin, NS, true, false>);
    return conv ? reinterpret_cast<const void*>(scan_bwd_kernel<Tin, NS, false, true>)
                : reinterpret_cast<const void*>(scan_bwd_kernel<Tin, NS, false, false>);
}

template <typename Tin>
const void* bwd_kernel_ptr_n(int N, int zoh, bool conv) {
    if (N <= 4) return bwd_kernel_ptr<Tin, 4>(zoh, conv);
    if (N <= 8) return bwd_kernel_ptr<Tin, 8>(zoh, conv);
    return bwd_kernel_ptr<Tin, 16>(zoh, conv);
}

int bwd_smem_n(int N) { return N <= 4 ? bwd_state_smem<4>() : N <= 8 ? bwd_state_smem<8>() : bwd_state_smem<16>(); }

}  // namespace

cudaError_t scan_bwd_resident_blocks(int dtype, int N, int zoh, bool conv, int* slots) {
    const void* k = dtype == 1 ? bwd_kernel_ptr_n<BF16>(N, zoh, conv) : bwd_kernel_ptr_n<F32>(N, zoh, conv);
    const cudaError_t e = set_dynamic_smem(k, bwd_smem_n(N));
    if (e != cudaSuccess) return e;
    return resident_blocks(k, kBwdThreads, bwd_smem_n(N), slots);
}

cudaError_t launch_scan_bwd(const ScanBwdArgs& a, int dtype, int zoh, cudaStream_t stream) {
    return dtype == 1 ? launch_bwd_t<BF16>(a, zoh, stream) : launch_bwd_t<F32>(a, zoh, stream);
}

}  // namespace ssm
