// Selective-scan kernel for bf16 inputs and outputs: four lanes per channel, tensor-core readout.
//
// Layout.  A warp owns 8 channels of one batch row.  Lane l works on channel g = l / 4 and keeps
// the fp32 states n = q + 4k (q = l % 4, k < NSL) in registers, so every lane still runs the plain
// time-sequential recurrence h_t = Abar h_{t-1} + Bbar v_t on its own states (dpshk.com/news/3333417
// sections 2.2/2.3; the diagonal A of section 3.2 decouples the states).  Small warps (8 channels)
// give 4x more warps than one-channel-per-lane and spread evenly over the 148 SMs.
//
// Readout.  y_t[g] = sum_n C_t[n] h_t[g, n] is a contraction over n of exactly the tensor-core
// m16n8k8 (tf32 in, fp32 accumulate) fragment shape: the A fragment of lane (g, q) is
// {h[g, q], 0, h[g, q+4], 0} per group of 8 states, the B fragment is {C_t[q], C_t[q+4]} in every
// column, so every column of row g of the result holds y_t[g].  The MMA replaces one fp32 FMA per
// (channel, state, step) on the FMA pipe, the scan's bottleneck.  h is rounded to tf32 (10-bit
// mantissa) for the readout only; the recurrence itself stays in fp32.  Used for bf16 outputs.
//
// Per-step scalars.  For each group of 8 steps, lane q computes the conv front end, softplus and gate
// for steps 2q, 2q+1 of its channel and shares (dt, v) through a per-warp shared-memory slot; the
// readout of step j lands in every lane and lane j/2 keeps it, so the D skip and the gate are applied
// by the lane that computed that step's v and gate.
//
// Staging.  Per 32-step chunk, cp.async copies the block's u/x (with an 8-step halo for the conv),
// delta, z rows and the B/C rows into shared memory one chunk ahead (double buffer); B/C are then
// widened to fp32 in the order lane q reads them.  Outputs go through a shared tile and leave as
// coalesced 16-byte stores.  Requires L % 8 == 0 and 16-byte-aligned rows (the host checks).
#pragma once

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

constexpr int kG4Threads = 128;         // 4 warps
constexpr int kG4Chan = 32;             // channels per block (8 per warp)
constexpr int kG4Chunk = 32;            // steps per staged chunk
constexpr int kG4Halo = 8;              // x steps staged before the chunk (conv history)
constexpr int kG4Row = kG4Halo + kG4Chunk;  // staged row length in elements (80 B, bank-spread)
constexpr int kG4OutRow = kG4Chunk / 2 + 4; // output tile row in bf16x2 words (padded)
constexpr int kG4Segs = kG4Chunk / 8;      // 16-byte segments per staged row

template <int NSL>
struct G4Smem {
    uint16_t x[2][kG4Chan][kG4Row];      // bf16 u / x, steps c0-8 .. c0+31
    uint16_t dl[2][kG4Chan][kG4Row];     // bf16 delta at [8 + t - c0]
    uint16_t zz[2][kG4Chan][kG4Row];     // bf16 z at [8 + t - c0]
    uint16_t bcr[2][2][4 * NSL][kG4Chunk];  // raw bf16 B / C rows (n, t)
    float bc[2][kG4Chunk][4][NSL];       // fp32: bc[w][t][q][k] = (B|C)_t[q + 4k]
    float4 xch[4][8][9];                 // per warp: (dt, dt, v, v) of channel g, step j (row padded)
    uint32_t ys[kG4Chan][kG4OutRow];     // bf16x2 output tile (read before, written after a barrier)
    float4 chw[kG4Chan];                 // per channel: conv taps w[0..3] (w[3] multiplies x_t)
    float4 chs[kG4Chan];                 // per channel: (conv bias, D skip, dt bias, 0)
};

// 7 resident blocks of 4 warps per SM (28 warps) fit the 4096 warps of a batch-8, 4096-channel
// problem in one round; that needs <= 31.5 KB of shared memory per block for N <= 16.
static_assert(sizeof(G4Smem<4>) <= 32256, "N <= 16 scan blocks must fit 7 per SM");

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    const int n = valid ? 16 : 0;  // 0: fill the 16 bytes with zeros, read nothing
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// m16n8k8 tf32 MMA, fp32 accumulate: d = a * b + c.
__device__ __forceinline__ void mma_tf32(float& d0, float& d1, float& d2, float& d3, float a0, float a2, float b0,
                                         float b1, float c0, float c1, float c2, float c3) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d0), "=f"(d1), "=f"(d2), "=f"(d3)
        : "r"(__float_as_uint(a0)), "r"(0u), "r"(__float_as_uint(a2)), "r"(0u), "r"(__float_as_uint(b0)),
          "r"(__float_as_uint(b1)), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

// Per-lane constants.  State pair p holds states (q + 8p, q + 8p + 4) of the lane's channel, the
// two states one tensor-core k-block takes from this lane.
template <int NSL>
struct G4Consts {
    f32x2 al2[NSL / 2];    // A * log2(e)
    f32x2 ninva[NSL / 2];  // -1 / A (0 where A == 0 or the state is padding; padding has B = C = 0)
};

// One group of 8 steps starting at chunk column j0 (all 8 steps lie inside [t_begin, t_end)).
template <int NSL, Disc kDisc, bool kFinal, bool kConv>
__device__ __forceinline__ void g4_group(const ScanKernelArgs& a, G4Smem<NSL>& sm, int buf, int warp, int g, int q,
                                         int cl, int j0, const G4Consts<NSL>& cc, f32x2 (&hp)[NSL / 2], float& dsum,
                                         bool has_z) {
    // --- per-step scalars for steps j0 + 2q, j0 + 2q + 1 of this lane's channel ---
    const int col = kG4Halo + j0 + 2 * q;
    const float4 chs = sm.chs[cl];  // (conv bias, D skip, dt bias, 0)
    const uint32_t xw = *reinterpret_cast<const uint32_t*>(&sm.x[buf][cl][col]);
    float v0, v1;
    if (kConv) {
        const float4 w = sm.chw[cl];
        const uint32_t xm4 = *reinterpret_cast<const uint32_t*>(&sm.x[buf][cl][col - 4]);
        const uint32_t xm2 = *reinterpret_cast<const uint32_t*>(&sm.x[buf][cl][col - 2]);
        const float x_3 = bf16_hi(xm4), x_2 = bf16_lo(xm2), x_1 = bf16_hi(xm2), x0 = bf16_lo(xw), x1 = bf16_hi(xw);
        float c0 = fmaf(w.x, x_3, chs.x), c1 = fmaf(w.x, x_2, chs.x);
        c0 = fmaf(w.y, x_2, c0); c1 = fmaf(w.y, x_1, c1);
        c0 = fmaf(w.z, x_1, c0); c1 = fmaf(w.z, x0, c1);
        c0 = fmaf(w.w, x0, c0);  c1 = fmaf(w.w, x1, c1);
        v0 = silu_fast(c0);
        v1 = silu_fast(c1);
    } else {
        v0 = bf16_lo(xw);
        v1 = bf16_hi(xw);
    }
    const uint32_t dw = *reinterpret_cast<const uint32_t*>(&sm.dl[buf][cl][col]);
    float dt0 = bf16_lo(dw) + chs.z, dt1 = bf16_hi(dw) + chs.z;
    if (a.softplus) {
        dt0 = softplus_fast(dt0);
        dt1 = softplus_fast(dt1);
    }
    float gate0 = 1.0f, gate1 = 1.0f;
    if (kFinal && has_z) {
        const uint32_t zw = *reinterpret_cast<const uint32_t*>(&sm.zz[buf][cl][col]);
        gate0 = silu_fast(bf16_lo(zw));
        gate1 = silu_fast(bf16_hi(zw));
    }

    // --- share (dt, v) of the 8 steps among the 4 lanes of the channel ---
    __syncwarp();
    sm.xch[warp][g][2 * q] = make_float4(dt0, dt0, v0, v0);
    sm.xch[warp][g][2 * q + 1] = make_float4(dt1, dt1, v1, v1);
    __syncwarp();

    // --- the recurrence (packed pairs of states) and the tensor-core readout, step by step ---
    // unrolled by 2 only: with 28 resident warps per SM the kernel has 72 registers per thread, and a
    // full unroll of the 8 steps spills.
    float y0 = 0.0f, y1 = 0.0f;
#pragma unroll 2
    for (int j = 0; j < 8; ++j) {
        const ulonglong2 dv = *reinterpret_cast<const ulonglong2*>(&sm.xch[warp][g][j]);
        const f32x2 dt2 = dv.x, v2 = dv.y;
        f32x2 Bp[NSL / 2], Cp[NSL / 2];
#pragma unroll
        for (int k4 = 0; k4 < NSL; k4 += 4) {
            const ulonglong2 bq = *reinterpret_cast<const ulonglong2*>(&sm.bc[0][j0 + j][q][k4]);
            Bp[k4 / 2] = bq.x;
            Bp[k4 / 2 + 1] = bq.y;
            if (kFinal) {
                const ulonglong2 cq = *reinterpret_cast<const ulonglong2*>(&sm.bc[1][j0 + j][q][k4]);
                Cp[k4 / 2] = cq.x;
                Cp[k4 / 2 + 1] = cq.y;
            }
        }
        if (kDisc == Disc::kSimple) {
            const f32x2 dv2 = mul2(dt2, v2);
#pragma unroll
            for (int p = 0; p < NSL / 2; ++p)
                hp[p] = fma2(ex2x2(mul2(dt2, cc.al2[p])), hp[p], mul2(dv2, Bp[p]));
        } else if (kDisc == Disc::kZOH) {
            // h' = Abar (h + g) - g with g = (v / a) B, written with ng = -g = (v * (-1/a)) B
#pragma unroll
            for (int p = 0; p < NSL / 2; ++p) {
                const f32x2 ab = ex2x2(mul2(dt2, cc.al2[p]));
                const f32x2 ng = mul2(mul2(v2, cc.ninva[p]), Bp[p]);
                hp[p] = fma2(ab, sub2(hp[p], ng), ng);
            }
        } else {  // exact: h' = Abar h + E v B (E from the series where |dt a| < 2^-4; dt at a = 0)
#pragma unroll
            for (int p = 0; p < NSL / 2; ++p) {
                const f32x2 y2 = mul2(dt2, cc.al2[p]);
                const f32x2 ab = ex2x2(y2);
                const f32x2 E = zoh_factor2(dt2, y2, ab, cc.ninva[p]);
                hp[p] = fma2(ab, hp[p], mul2(E, mul2(v2, Bp[p])));
            }
        }
        if (kFinal) {
            float d0 = 0.0f, d1 = 0.0f, d2 = 0.0f, d3 = 0.0f;
#pragma unroll
            for (int p = 0; p < NSL / 2; ++p) {
                float a0, a2, b0, b1;
                unpack2(hp[p], a0, a2);
                unpack2(Cp[p], b0, b1);
                mma_tf32(d0, d1, d2, d3, a0, a2, b0, b1, d0, d1, d2, d3);
            }
            if ((j >> 1) == q) {
                if (j & 1) y1 = d0;
                else y0 = d0;
            }
        } else {
            float dtj, dtj2;
            unpack2(dt2, dtj, dtj2);
            dsum += dtj;
        }
    }

    if (kFinal) {
        const float dskip = sm.chs[cl].y;
        const float o0 = fmaf(dskip, sm.xch[warp][g][2 * q].z, y0) * gate0;
        const float o1 = fmaf(dskip, sm.xch[warp][g][2 * q + 1].z, y1) * gate1;
        sm.ys[cl][(j0 >> 1) + q] = pack_bf16x2(o0, o1);
    }
}

// Copies one chunk (steps c0 .. c0+63 plus the x halo) of the block's rows into buffer `buf`.
template <int NSL>
__device__ __forceinline__ void g4_issue_chunk(const ScanKernelArgs& a, G4Smem<NSL>& sm, int buf, int b, int ch0,
                                               int c0, bool want_z) {
    const int tid = threadIdx.x;
    const uint16_t* u = static_cast<const uint16_t*>(a.u);
    const uint16_t* dl = static_cast<const uint16_t*>(a.delta);
    const uint16_t* zz = static_cast<const uint16_t*>(a.z);
    // x / u: 32 rows x (1 + kG4Segs) segments of 8 steps (the first is the halo)
    for (int i = tid; i < kG4Chan * (kG4Segs + 1); i += kG4Threads) {
        const int r = i / (kG4Segs + 1), s = i - r * (kG4Segs + 1);
        const int d = ch0 + r;
        const int t = c0 - kG4Halo + 8 * s;
        const bool ok = d < a.D && t >= 0 && t < a.L;
        const uint16_t* src = ok ? u + ((size_t)b * a.D + d) * a.L + t : u;
        cp_async16(&sm.x[buf][r][8 * s], src, ok);
    }
    for (int i = tid; i < kG4Chan * kG4Segs; i += kG4Threads) {
        const int r = i / kG4Segs, s = i % kG4Segs;
        const int d = ch0 + r;
        const int t = c0 + 8 * s;
        const bool ok = d < a.D && t < a.L;
        const size_t off = ((size_t)b * a.D + d) * a.L + t;
        cp_async16(&sm.dl[buf][r][kG4Halo + 8 * s], ok ? dl + off : dl, ok);
        if (want_z) cp_async16(&sm.zz[buf][r][kG4Halo + 8 * s], ok ? zz + off : zz, ok);
    }
    // B / C: N rows x kG4Segs segments each (rows past N stay zero from the initial clear)
    const uint16_t* Bm = static_cast<const uint16_t*>(a.Bm);
    const uint16_t* Cm = static_cast<const uint16_t*>(a.Cm);
    for (int i = tid; i < 2 * a.N * kG4Segs; i += kG4Threads) {
        const int w = i / (a.N * kG4Segs);
        const int rem = i - w * a.N * kG4Segs;
        const int n = rem / kG4Segs, s = rem % kG4Segs;
        const int t = c0 + 8 * s;
        const bool ok = t < a.L;
        const size_t off = ((size_t)b * a.N + n) * a.L + t;
        const uint16_t* base = w ? Cm : Bm;
        cp_async16(&sm.bcr[buf][w][n][8 * s], ok ? base + off : base, ok);
    }
    cp_async_commit();
}

template <int NSL, bool kZOH, bool kFinal, bool kConv>
__global__ void __launch_bounds__(kG4Threads, 7) scan_g4_kernel(const ScanKernelArgs a) {
    extern __shared__ __align__(16) unsigned char g4_smem_raw[];
    G4Smem<NSL>& sm = *reinterpret_cast<G4Smem<NSL>*>(g4_smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;
    const int b = blockIdx.y, seg = blockIdx.z;
    const int ch0 = blockIdx.x * kG4Chan;
    const int cl = warp * 8 + g;
    const int d = ch0 + cl;
    const bool active = d < a.D;
    const size_t rows = (size_t)a.Bsz * a.D;
    const size_t row = (size_t)b * a.D + (active ? d : 0);
    const int t_begin = seg * a.seg_len;
    const int t_end = min(a.L, t_begin + a.seg_len);
    const bool has_z = kFinal && a.z != nullptr;

    // zero the B/C raw rows past N once (cp.async never writes them)
    for (int i = tid; i < 2 * 2 * 4 * NSL * kG4Chunk; i += kG4Threads) (&sm.bcr[0][0][0][0])[i] = 0;
    __syncthreads();
    g4_issue_chunk<NSL>(a, sm, 0, b, ch0, t_begin, has_z);

    G4Consts<NSL> cc;
    bool small_a = false;  // some state with |A| < kZohFastMinA (0 included): the exact form
#pragma unroll
    for (int p = 0; p < NSL / 2; ++p) {
        float al[2], ni[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int n = q + 4 * (2 * p + e);
            const bool real = active && n < a.N;
            const float av = real ? __ldg(a.A + (size_t)d * a.N + n) : 0.0f;
            al[e] = av * kLog2e;
            ni[e] = av != 0.0f ? -1.0f / av : 0.0f;
            small_a |= real && !(fabsf(av) >= kZohFastMinA);
        }
        cc.al2[p] = pack2(al[0], al[1]);
        cc.ninva[p] = pack2(ni[0], ni[1]);
    }
    if (q == 0) {  // per-channel scalars, read once per 8-step group from shared memory
        float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
        float cb = 0.0f;
        if (kConv && active) {
            const int W = a.conv_width;
            const float* cw = a.conv_w + (size_t)d * W;
            // tap i of the 4-wide window is tap i - (4 - W) of the filter
            w.x = W >= 4 ? __ldg(cw + 0 - (4 - W)) : 0.0f;
            w.y = W >= 3 ? __ldg(cw + 1 - (4 - W)) : 0.0f;
            w.z = W >= 2 ? __ldg(cw + 2 - (4 - W)) : 0.0f;
            w.w = __ldg(cw + 3 - (4 - W));
            if (a.conv_b != nullptr) cb = __ldg(a.conv_b + d);
        }
        sm.chw[cl] = w;
        sm.chs[cl] = make_float4(cb, (a.Dskip != nullptr && active) ? __ldg(a.Dskip + d) : 0.0f,
                                 (a.delta_bias != nullptr && active) ? __ldg(a.delta_bias + d) : 0.0f, 0.0f);
    }

    float h[NSL];
#pragma unroll
    for (int k = 0; k < NSL; ++k) h[k] = 0.0f;
    float dsum = 0.0f;
    if (kFinal) {
        const float* h0 = (a.nseg > 1) ? a.ws_h0 : a.h0;
        if (h0 != nullptr && active) {
#pragma unroll
            for (int k = 0; k < NSL; ++k)
                if (q + 4 * k < a.N) h[k] = h0[row * a.N + q + 4 * k];
        }
        for (int s = 0; s < seg; ++s) {
            const float S = active ? a.ws_dsum[(size_t)s * rows + row] : 0.0f;
#pragma unroll
            for (int k = 0; k < NSL; ++k) {
                const int n = q + 4 * k;
                float al0, al1;
                unpack2(cc.al2[k / 2], al0, al1);
                const float hs = (active && n < a.N) ? a.ws_h[((size_t)s * rows + row) * a.N + n] : 0.0f;
                h[k] = fmaf(ex2((k & 1 ? al1 : al0) * S), h[k], hs);
            }
        }
    } else if (seg == 0 && a.ws_h0 != nullptr && a.h0 != nullptr && active) {
#pragma unroll
        for (int k = 0; k < NSL; ++k)
            if (q + 4 * k < a.N) a.ws_h0[row * a.N + q + 4 * k] = a.h0[row * a.N + q + 4 * k];
    }
    f32x2 hp[NSL / 2];
#pragma unroll
    for (int p = 0; p < NSL / 2; ++p) hp[p] = pack2(h[2 * p], h[2 * p + 1]);
    const bool exact = kZOH && __any_sync(0xffffffffu, small_a);  // warp-uniform choice of loop body

    int buf = 0;
    for (int c0 = t_begin; c0 < t_end; c0 += kG4Chunk, buf ^= 1) {
        cp_async_wait_all();
        __syncthreads();  // chunk c0 landed for every thread; everyone is done with the other buffers
        if (kFinal && c0 > t_begin) {
            // store the previous chunk's output tile, 16 bytes per thread-op; every read of the tile
            // happens before the barrier below, every write of the next tile after it
            const int pc0 = c0 - kG4Chunk;
            uint16_t* y = static_cast<uint16_t*>(a.y);
            for (int i = tid; i < kG4Chan * kG4Segs; i += kG4Threads) {
                const int r = i / kG4Segs, s = i % kG4Segs;
                const int dd = ch0 + r, t = pc0 + 8 * s;
                if (dd < a.D && t < t_end) {
                    const uint4 w = *reinterpret_cast<const uint4*>(&sm.ys[r][4 * s]);
                    __stcs(reinterpret_cast<uint4*>(y + ((size_t)b * a.D + dd) * a.L + t), w);
                }
            }
        }
        if (c0 + kG4Chunk < t_end) g4_issue_chunk<NSL>(a, sm, buf ^ 1, b, ch0, c0 + kG4Chunk, has_z);
        if (kConv && c0 == 0 && a.conv_init != nullptr) {
            // x before t = 0 is the caller's history (oldest first), not the zeros the copy filled in
            const int W1 = a.conv_width - 1;
            for (int i = tid; i < kG4Chan * W1; i += kG4Threads) {
                const int r = i / W1, k = i - r * W1;
                if (ch0 + r < a.D)
                    sm.x[buf][r][kG4Halo - W1 + k] =
                        static_cast<const uint16_t*>(a.conv_init)[((size_t)b * a.D + ch0 + r) * W1 + k];
            }
        }
        // widen B / C of this chunk to fp32, in lane order
        for (int i = tid; i < 2 * kG4Chunk * 4; i += kG4Threads) {
            const int w = i / (kG4Chunk * 4);
            const int rem = i - w * kG4Chunk * 4;
            const int t = rem >> 2, qq = rem & 3;
#pragma unroll
            for (int k4 = 0; k4 < NSL; k4 += 4) {
                float4 f;
                f.x = bf16_to_f32(sm.bcr[buf][w][qq + 4 * k4][t]);
                f.y = bf16_to_f32(sm.bcr[buf][w][qq + 4 * (k4 + 1)][t]);
                f.z = bf16_to_f32(sm.bcr[buf][w][qq + 4 * (k4 + 2)][t]);
                f.w = bf16_to_f32(sm.bcr[buf][w][qq + 4 * (k4 + 3)][t]);
                *reinterpret_cast<float4*>(&sm.bc[w][t][qq][k4]) = f;
            }
        }
        __syncthreads();
        const int clen = min(kG4Chunk, t_end - c0);
        for (int j0 = 0; j0 < clen; j0 += 8) {
            if (exact)
                g4_group<NSL, Disc::kZOHExact, kFinal, kConv>(a, sm, buf, warp, g, q, cl, j0, cc, hp, dsum, has_z);
            else
                g4_group<NSL, kZOH ? Disc::kZOH : Disc::kSimple, kFinal, kConv>(a, sm, buf, warp, g, q, cl, j0, cc, hp,
                                                                              dsum, has_z);
        }
    }
    if (kFinal) {
        __syncthreads();
        const int nch = (t_end - t_begin + kG4Chunk - 1) / kG4Chunk;
        const int pc0 = t_begin + (nch - 1) * kG4Chunk;
        uint16_t* y = static_cast<uint16_t*>(a.y);
        for (int i = tid; i < kG4Chan * kG4Segs; i += kG4Threads) {
            const int r = i / kG4Segs, s = i % kG4Segs;
            const int dd = ch0 + r, t = pc0 + 8 * s;
            if (dd < a.D && t < t_end) {
                const uint4 w = *reinterpret_cast<const uint4*>(&sm.ys[r][4 * s]);
                __stcs(reinterpret_cast<uint4*>(y + ((size_t)b * a.D + dd) * a.L + t), w);
            }
        }
    }
    if (!active) return;
#pragma unroll
    for (int p = 0; p < NSL / 2; ++p) unpack2(hp[p], h[2 * p], h[2 * p + 1]);
    if (kFinal) {
        if (seg == a.nseg - 1 && a.h_out != nullptr) {
#pragma unroll
            for (int k = 0; k < NSL; ++k)
                if (q + 4 * k < a.N) a.h_out[row * a.N + q + 4 * k] = h[k];
        }
    } else {
        if (q == 0) a.ws_dsum[(size_t)seg * rows + row] = dsum;
#pragma unroll
        for (int k = 0; k < NSL; ++k)
            if (q + 4 * k < a.N) a.ws_h[((size_t)seg * rows + row) * a.N + q + 4 * k] = h[k];
    }
}

template <int NSL, bool kZOH, bool kConv>
cudaError_t launch_g4_ns(const ScanKernelArgs& a, cudaStream_t stream) {
    const size_t smem = sizeof(G4Smem<NSL>);
    dim3 block(kG4Threads);
    const unsigned gx = (unsigned)((a.D + kG4Chan - 1) / kG4Chan);
    cudaError_t e;
    if (a.nseg > 1) {
        auto kfn = scan_g4_kernel<NSL, kZOH, false, kConv>;
        e = set_dynamic_smem_once(kfn, (int)smem);
        if (e != cudaSuccess) return e;
        kfn<<<dim3(gx, (unsigned)a.Bsz, (unsigned)(a.nseg - 1)), block, smem, stream>>>(a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    auto kfn = scan_g4_kernel<NSL, kZOH, true, kConv>;
    e = set_dynamic_smem_once(kfn, (int)smem);
    if (e != cudaSuccess) return e;
    kfn<<<dim3(gx, (unsigned)a.Bsz, (unsigned)a.nseg), block, smem, stream>>>(a);
    return cudaGetLastError();
}

template <int NSL>
cudaError_t launch_g4_nsl(const ScanKernelArgs& a, int zoh, cudaStream_t s) {
    const bool conv = a.conv_w != nullptr;
    if (zoh) return conv ? launch_g4_ns<NSL, true, true>(a, s) : launch_g4_ns<NSL, true, false>(a, s);
    return conv ? launch_g4_ns<NSL, false, true>(a, s) : launch_g4_ns<NSL, false, false>(a, s);
}

}  // namespace ssm
