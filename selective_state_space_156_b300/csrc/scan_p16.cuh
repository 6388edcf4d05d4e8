// Selective-scan kernel for aligned bf16 problems: LPC lanes per channel, packed fp32 pairs.
//
// Layout.  A block of 128 threads owns 128 / LPC channels of one batch row and one L segment.  The
// LPC lanes of a channel each keep N / LPC of its fp32 states in registers and walk the segment in
// time order, so the recurrence h_t = Abar h_{t-1} + Bbar v_t (dpshk.com/news/3333417 sections
// 2.2/2.3; the diagonal A of section 3.2 decouples the states) needs no exchange between lanes; only
// the readout y = sum_n C h is summed over the LPC lanes with xor shuffles.  LPC trades per-step
// overhead (shared by N / LPC states per lane) against warps per SM (latency hiding): the host picks it
// from the problem size.  The state update and the readout run on pairs of states with the sm_100+
// packed f32x2 instructions: one issue slot per two lanes of FMA work.
//
// Per-step scalars.  Within a group of 8 steps, lane e of a channel computes the conv front end,
// softplus and gate of steps [e 8/LPC, (e+1) 8/LPC); the (dt, v) of the other steps come from the
// owning lanes by shuffle, and each lane applies the D skip and gate to, and stores, its own steps.
//
// Zero-order hold per state pair, with ninv = -1/a and ng = (v ninv) B = -(v/a) B:
//   h' = Abar (h - ng) + ng  ==  Abar h + (Abar - 1)(v/a) B,
// whose fixed point for a constant input is -ng exactly, whatever the rounding of Abar.  Its error per
// step grows as |v B / a|, so a block in which some state has |a| < kZohFastMinA (a == 0 included) runs
// a second loop body, h' = Abar h + E v B with E = (exp(dt a) - 1) / a from zoh_factor2 (a Taylor series
// where |dt a| is small, the limit dt at a = 0; lshu.cn/news/79586 2.2).
//
// Staging.  Per 48-step chunk, five tiled bulk tensor copies (TMA, issued by one thread, completing on
// an mbarrier) bring the block's u/x rows (with an 8-step halo for the conv front end of
// dpshk.com/news/3333417 section 5.2), delta and z rows and the B/C rows of the batch row into shared
// memory one chunk ahead (double buffer); per-thread cp.async copies remain as the alternative.  B/C
// are widened to fp32 once per chunk and read by every lane as broadcasts.  Outputs leave as 16-byte stores of 8 steps.  Requires L % 8 == 0 and
// 16-byte-aligned rows (the host checks).  bf16 outputs use MUFU tanh/lg2 forms of SiLU and softplus.
#pragma once

#include <cstdlib>
#include <cstring>

#include "ssm_device.cuh"
#include "ssm_internal.h"
#include "tma.cuh"

namespace ssm {

constexpr int kP16Threads = 128;              // threads per block
constexpr int kP16Chunk = 48;                 // steps per staged chunk
constexpr int kP16Halo = 8;                   // x steps staged before the chunk (conv history)
constexpr int kP16Row = kP16Halo + kP16Chunk; // staged row length in elements (112 B)
constexpr int kP16Segs = kP16Chunk / 8;       // 16-byte segments per staged row

template <int NS, int LPC>
struct P16Smem {
    static constexpr int kCh = kP16Threads / LPC;  // channels per block
    static constexpr int kNSR = NS < 8 ? 8 : NS;   // B / C rows per block of bcr: a multiple of 128 bytes
    // every tile that a bulk tensor copy fills starts on a 128-byte boundary (rows of 112 bytes: 8 rows
    // = 896 bytes, and kCh, kNSR are multiples of 8)
    uint16_t x[2][kCh][kP16Row];               // bf16 u / x, steps c0-8 .. c0+31
    uint16_t dl[2][kCh][kP16Row];              // bf16 delta at [8 + t - c0]
    uint16_t zz[2][kCh][kP16Row];              // bf16 z at [8 + t - c0]
    uint16_t bcr[2][2][kNSR][kP16Row];         // raw bf16 B / C rows (n, t), padded against bank conflicts
    float bc[kP16Chunk][2][NS];                // fp32 B_t[n], C_t[n]
    uint64_t bar[2];                           // mbarriers of the two chunk buffers (bulk-copy staging)
};

__device__ __forceinline__ void p16_cp_async16(void* smem, const void* gmem, bool valid) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    const int n = valid ? 16 : 0;  // 0: fill the 16 bytes with zeros, read nothing
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}

// Tensor maps of the tiled bulk copies (TMA) that stage a chunk: x (with the conv halo), delta, z as
// (L, B*D) matrices with boxes of 40 steps x the block's channels, B and C as (L, B*N) matrices with
// boxes of 40 steps x NS states.  Every box starts 8 steps before the chunk, so the staged rows have
// the layout of the per-thread copies below (the chunk at column 8); rows past the matrix come in as
// zeros, and B / C rows of the next batch row (n >= N) are masked when they are widened.
struct P16Maps {
    CUtensorMap x, dl, zz, B, C;
};

// Set when a wait for a chunk's copies ran out (about a second): the block then leaves its outputs
// unwritten.  Read and cleared by take_scan_wait_error (ssm_device_error).
static __device__ unsigned int g_scan_wait_error = 0;

template <int NS, int LPC>
__device__ __forceinline__ void p16_tma_chunk(const P16Maps& maps, P16Smem<NS, LPC>& sm, uint64_t* bar, int buf,
                                              int row0, int brow0, int c0, bool want_z) {
    constexpr int kCh = P16Smem<NS, LPC>::kCh;
    constexpr unsigned kRowBytes = kP16Row * 2;
    const unsigned bytes = kRowBytes * (2u * kCh + (want_z ? kCh : 0u) + 2u * NS);
    mbar_arrive_expect_tx(bar, bytes);
    tma_load_2d(&sm.x[buf][0][0], &maps.x, c0 - kP16Halo, row0, bar);
    tma_load_2d(&sm.dl[buf][0][0], &maps.dl, c0 - kP16Halo, row0, bar);
    if (want_z) tma_load_2d(&sm.zz[buf][0][0], &maps.zz, c0 - kP16Halo, row0, bar);
    tma_load_2d(&sm.bcr[buf][0][0][0], &maps.B, c0 - kP16Halo, brow0, bar);
    tma_load_2d(&sm.bcr[buf][1][0][0], &maps.C, c0 - kP16Halo, brow0, bar);
}

template <int NS, int LPC>
__device__ __forceinline__ void p16_issue_chunk(const ScanKernelArgs& a, P16Smem<NS, LPC>& sm, int buf, int b, int ch0,
                                                int c0, bool want_z) {
    constexpr int kCh = P16Smem<NS, LPC>::kCh;
    const int tid = threadIdx.x;
    const uint16_t* u = static_cast<const uint16_t*>(a.u);
    const uint16_t* dl = static_cast<const uint16_t*>(a.delta);
    const uint16_t* zz = static_cast<const uint16_t*>(a.z);
    const bool conv = a.conv_w != nullptr;
    // rows of u / x: the halo segment only when the conv needs it
    for (int i = tid; i < kCh * (kP16Segs + 1); i += kP16Threads) {
        const int r = i / (kP16Segs + 1), s = i - r * (kP16Segs + 1);
        if (s == 0 && !conv) continue;
        const int d = ch0 + r;
        const int t = c0 - kP16Halo + 8 * s;
        const bool ok = d < a.D && t >= 0 && t < a.L;
        p16_cp_async16(&sm.x[buf][r][8 * s], ok ? u + ((size_t)b * a.D + d) * a.L + t : u, ok);
    }
    for (int i = tid; i < kCh * kP16Segs; i += kP16Threads) {
        const int r = i / kP16Segs, s = i - r * kP16Segs;
        const int d = ch0 + r;
        const int t = c0 + 8 * s;
        const bool ok = d < a.D && t < a.L;
        const size_t off = ((size_t)b * a.D + d) * a.L + t;
        p16_cp_async16(&sm.dl[buf][r][kP16Halo + 8 * s], ok ? dl + off : dl, ok);
        if (want_z) p16_cp_async16(&sm.zz[buf][r][kP16Halo + 8 * s], ok ? zz + off : zz, ok);
    }
    const uint16_t* Bm = static_cast<const uint16_t*>(a.Bm);
    const uint16_t* Cm = static_cast<const uint16_t*>(a.Cm);
    for (int i = tid; i < 2 * a.N * kP16Segs; i += kP16Threads) {
        const int w = i / (a.N * kP16Segs);
        const int rem = i - w * a.N * kP16Segs;
        const int n = rem / kP16Segs, s = rem - n * kP16Segs;
        const int t = c0 + 8 * s;
        const bool ok = t < a.L;
        const uint16_t* base = w ? Cm : Bm;
        p16_cp_async16(&sm.bcr[buf][w][n][8 * s], ok ? base + ((size_t)b * a.N + n) * a.L + t : base, ok);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Per-lane constants: lane e of a channel holds states [e NSL, (e+1) NSL); pair p = states (2p, 2p+1)
// of that range.
template <int NSL>
struct P16Consts {
    f32x2 al2[NSL / 2];   // A log2(e)
    f32x2 ninv[NSL / 2];  // -1/A (0 where A == 0 or padding; padding has B = C = 0)
};

// 8 steps starting at chunk column j0 (all inside [t_begin, t_end)).
template <int NS, int LPC, Disc kDisc, bool kFinal, bool kConv, bool kHall>
__device__ __forceinline__ void p16_group(const ScanKernelArgs& a, const P16Smem<NS, LPC>& sm, int buf, int j0,
                                          const P16Consts<NS / LPC>& cc, const float (&w)[4], float cb, float dskip,
                                          float bias, f32x2 (&hp)[NS / LPC / 2], float& dsum, bool has_z,
                                          bool active, size_t yoff, float* hall) {
    constexpr int NSL = NS / LPC;   // states per lane
    constexpr int SPL = 8 / LPC;    // steps whose scalars this lane owns
    const int lane = threadIdx.x & 31;
    const int e = lane & (LPC - 1);
    const int r = threadIdx.x / LPC;          // channel within the block
    const int src0 = lane & ~(LPC - 1);       // first lane of this channel
    const int col = kP16Halo + j0 + e * SPL;  // first owned step's column
    // --- scalars of the owned steps: SSM input v (conv front end), step dt, gate ---
    float xs[SPL], v[SPL], dto[SPL], gate[SPL];
    const uint16_t* xrow = &sm.x[buf][r][col];
#pragma unroll
    for (int k = 0; k < SPL; k += 2) {
        const uint32_t xw = *reinterpret_cast<const uint32_t*>(xrow + k);
        xs[k] = bf16_lo(xw);
        xs[k + 1] = bf16_hi(xw);
    }
    if (kConv) {
        // two 4-byte reads: the owned steps start at an even column, not always at a multiple of 4
        const uint32_t hw0 = *reinterpret_cast<const uint32_t*>(xrow - 4);
        const uint32_t hw1 = *reinterpret_cast<const uint32_t*>(xrow - 2);
        const float h3 = bf16_hi(hw0), h2 = bf16_lo(hw1), h1 = bf16_hi(hw1);  // x_{t-3}, x_{t-2}, x_{t-1}
#pragma unroll
        for (int k = 0; k < SPL; ++k) {
            const float xm3 = k >= 3 ? xs[k - 3] : (k == 0 ? h3 : (k == 1 ? h2 : h1));
            const float xm2 = k >= 2 ? xs[k - 2] : (k == 0 ? h2 : h1);
            const float xm1 = k >= 1 ? xs[k - 1] : h1;
            float c = fmaf(w[0], xm3, cb);
            c = fmaf(w[1], xm2, c);
            c = fmaf(w[2], xm1, c);
            c = fmaf(w[3], xs[k], c);
            v[k] = fmaf(c, tanh_mufu(c), c);  // SiLU(2c) = c + c tanh(c): the taps and bias are pre-halved
        }
    } else {
#pragma unroll
        for (int k = 0; k < SPL; ++k) v[k] = xs[k];
    }
    {
        // branch-free (compute, then select): the group stays one basic block, so the scheduler can
        // overlap these MUFU-heavy scalars with the FMA-heavy steps below
        const uint16_t* drow = &sm.dl[buf][r][col];
        const bool sp_on = a.softplus != 0;
#pragma unroll
        for (int k = 0; k < SPL; k += 2) {
            const uint32_t dw = *reinterpret_cast<const uint32_t*>(drow + k);
            if (kDisc == Disc::kZOH) {
                // the fast form needs the step only as the exponent argument dt a log2 e: keep it in base-2
                // units, t = dt log2 e = max(s', 0) + log2(1 + 2^-|s'|) with s' = s log2 e (bias pre-scaled),
                // and multiply by a (not a log2 e) below
                const float s0 = fmaf(bf16_lo(dw), kLog2e, bias), s1 = fmaf(bf16_hi(dw), kLog2e, bias);
                const float p0 = fmaxf(s0, 0.0f) + lg2_mufu(1.0f + ex2(-fabsf(s0)));
                const float p1 = fmaxf(s1, 0.0f) + lg2_mufu(1.0f + ex2(-fabsf(s1)));
                dto[k] = sp_on ? p0 : s0;
                dto[k + 1] = sp_on ? p1 : s1;
            } else {
                const float s0 = bf16_lo(dw) + bias, s1 = bf16_hi(dw) + bias;
                const float p0 = softplus_fast(s0), p1 = softplus_fast(s1);
                dto[k] = sp_on ? p0 : s0;
                dto[k + 1] = sp_on ? p1 : s1;
            }
        }
    }
    if (kFinal) {
        // without z the staged z rows hold stale values; the select (not a product) keeps them out
        const uint16_t* zrow = &sm.zz[buf][r][col];
#pragma unroll
        for (int k = 0; k < SPL; k += 2) {
            const uint32_t zw = *reinterpret_cast<const uint32_t*>(zrow + k);
            const float g0 = silu_fast(bf16_lo(zw)), g1 = silu_fast(bf16_hi(zw));
            gate[k] = has_z ? g0 : 1.0f;
            gate[k + 1] = has_z ? g1 : 1.0f;
        }
    }

    // --- the recurrence and the readout, step by step ---
    float out[SPL];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float dtj, vj;
        if (LPC == 1) {
            dtj = dto[j];
            vj = v[j];
        } else {  // step j's scalars live in lane src0 + j / SPL, register j % SPL
            dtj = __shfl_sync(0xffffffffu, dto[j % SPL], src0 + j / SPL);
            vj = __shfl_sync(0xffffffffu, v[j % SPL], src0 + j / SPL);
        }
        const f32x2 dt2 = pack2(dtj, dtj);
        const f32x2 v2 = pack2(vj, vj);
        const float* Bt = sm.bc[j0 + j][0] + e * NSL;
        const float* Ct = sm.bc[j0 + j][1] + e * NSL;
        f32x2 Bp[NSL / 2], Cp[NSL / 2];
#pragma unroll
        for (int p4 = 0; p4 < NSL / 2; p4 += 2) {
            const ulonglong2 bq = *reinterpret_cast<const ulonglong2*>(Bt + 2 * p4);
            Bp[p4] = bq.x;
            Bp[p4 + 1] = bq.y;
            if (kFinal) {
                const ulonglong2 cq = *reinterpret_cast<const ulonglong2*>(Ct + 2 * p4);
                Cp[p4] = cq.x;
                Cp[p4 + 1] = cq.y;
            }
        }
        // in phases: every pair's exponent and Abar (MUFU), then the input terms, then the updates, so that
        // the MUFU results of the first pairs are ready when the FMA pipe reaches them (3 % faster than
        // one pair at a time on the 8 x 4096 x 16 x 2048 layer)
        f32x2 y2[NSL / 2], ab[NSL / 2];
#pragma unroll
        for (int p = 0; p < NSL / 2; ++p) {
            y2[p] = mul2(dt2, cc.al2[p]);
            ab[p] = ex2x2(y2[p]);
        }
        if (kDisc == Disc::kSimple) {
            const f32x2 dv2 = mul2(dt2, v2);
#pragma unroll
            for (int p = 0; p < NSL / 2; ++p) hp[p] = fma2(ab[p], hp[p], mul2(dv2, Bp[p]));
        } else if (kDisc == Disc::kZOH) {
            f32x2 ng[NSL / 2];
#pragma unroll
            for (int p = 0; p < NSL / 2; ++p) ng[p] = mul2(mul2(v2, cc.ninv[p]), Bp[p]);
#pragma unroll
            for (int p = 0; p < NSL / 2; ++p) hp[p] = fma2(ab[p], sub2(hp[p], ng[p]), ng[p]);
        } else {  // exact: h' = Abar h + E v B (E from the series where |dt a| < 2^-4; dt at a = 0)
#pragma unroll
            for (int p = 0; p < NSL / 2; ++p) {
                const f32x2 E = zoh_factor2(dt2, y2[p], ab[p], cc.ninv[p]);
                hp[p] = fma2(ab[p], hp[p], mul2(E, mul2(v2, Bp[p])));
            }
        }
        f32x2 acc = pack2(0.0f, 0.0f);
        if (kFinal) {
#pragma unroll
            for (int p = 0; p < NSL / 2; ++p) acc = fma2(Cp[p], hp[p], acc);
        }
        if (kHall && active && (a.hall_every <= 1 || j == 7)) {
            // the state after this step, into h_all (B, L, D, N), or after the group's last step into the
            // checkpoints (B, L / 8, D, N) (groups start at multiples of 8): this lane's states, 16-byte stores
            float* hp_out = hall + (size_t)(a.hall_every <= 1 ? j0 + j : j0 / 8) * a.D * a.N;
            if (a.N == NS) {
#pragma unroll
                for (int p = 0; p < NSL / 2; p += 2)
                    *reinterpret_cast<ulonglong2*>(hp_out + 2 * p) = make_ulonglong2(hp[p], hp[p + 1]);
            } else {
#pragma unroll
                for (int p = 0; p < NSL / 2; ++p) {
                    float h0_, h1_;
                    unpack2(hp[p], h0_, h1_);
                    if (e * NSL + 2 * p < a.N) hp_out[2 * p] = h0_;
                    if (e * NSL + 2 * p + 1 < a.N) hp_out[2 * p + 1] = h1_;
                }
            }
        }
        if (kFinal) {
            float ya, yb;
            unpack2(acc, ya, yb);
            float y = ya + yb;
#pragma unroll
            for (int m = 1; m < LPC; m <<= 1) y += __shfl_xor_sync(0xffffffffu, y, m);
            if (j / SPL == e) out[j % SPL] = y;
        } else {
            dsum += kDisc == Disc::kZOH ? dtj * kLn2 : dtj;  // the fast form's dtj is in base-2 units
        }
    }
    if (kFinal && active) {
#pragma unroll
        for (int k = 0; k < SPL; ++k) out[k] = fmaf(dskip, v[k], out[k]) * gate[k];
        uint16_t* y = static_cast<uint16_t*>(a.y) + yoff + j0 + e * SPL;
        if constexpr (SPL == 8) {
            store8<BF16>(a.y, yoff + j0, out);
        } else if constexpr (SPL == 4) {
            *reinterpret_cast<uint2*>(y) = make_uint2(pack_bf16x2(out[0], out[1]), pack_bf16x2(out[2], out[3]));
        } else {
            *reinterpret_cast<uint32_t*>(y) = pack_bf16x2(out[0], out[1]);
        }
    }
}

// Resident blocks per SM the register budget aims at, by lanes per channel.
__host__ __device__ constexpr int p16_min_blocks(int lpc) { return lpc == 1 ? 2 : (lpc == 2 ? 4 : 7); }

// One block's pass over segment `seg` of its (batch row, channel block): the final pass (outputs) or the
// summary pass (end state from a zero start and the sum of dt, for the L split).  kSeg0: the split has a
// first segment of its own length (a.seg0_len) whose final pass runs in the first launch; else the
// segments are [s seg_len, (s + 1) seg_len) (one of them when the sequence runs in one pass).
template <int NS, int LPC, bool kZOH, bool kFinal, bool kConv, bool kHall, bool kTma, bool kSeg0>
__device__ __forceinline__ void p16_run(const ScanKernelArgs& a, const P16Maps& maps, const int seg) {
    constexpr int NSL = NS / LPC;
    constexpr int kCh = P16Smem<NS, LPC>::kCh;
    constexpr int kBcOff = kTma ? kP16Halo : 0;  // column of the chunk's first step in the staged B / C rows
    extern __shared__ __align__(128) unsigned char p16_smem_raw[];
    P16Smem<NS, LPC>& sm = *reinterpret_cast<P16Smem<NS, LPC>*>(p16_smem_raw);
    uint64_t* tma_bar = sm.bar;
    const int tid = threadIdx.x;
    const int e = tid & (LPC - 1);
    const int b = blockIdx.y;
    const int ch0 = blockIdx.x * kCh;
    const int d = ch0 + tid / LPC;
    const bool active = d < a.D;
    const size_t rows = (size_t)a.Bsz * a.D;
    const size_t row = (size_t)b * a.D + (active ? d : 0);
    // segments: [s seg_len, (s + 1) seg_len), or with a first segment of seg0_len steps, [0, seg0_len) and
    // then seg_len steps each
    const int t_begin = kSeg0 ? (seg == 0 ? 0 : a.seg0_len + (seg - 1) * a.seg_len) : seg * a.seg_len;
    const int t_end = min(a.L, (kSeg0 && seg == 0) ? a.seg0_len : t_begin + a.seg_len);
    const bool has_z = kFinal && a.z != nullptr;

    // B/C rows past N stay zero (cp.async never writes them)
    for (int i = tid; i < 2 * 2 * P16Smem<NS, LPC>::kNSR * kP16Row; i += kP16Threads) (&sm.bcr[0][0][0][0])[i] = 0;
    const int row0 = b * a.D + ch0, brow0 = b * a.N;
    if (kTma && tid == 0) {
        tma_prefetch_map(&maps.x);
        tma_prefetch_map(&maps.dl);
        if (has_z) tma_prefetch_map(&maps.zz);
        tma_prefetch_map(&maps.B);
        tma_prefetch_map(&maps.C);
        mbar_init(&tma_bar[0], 1);
        mbar_init(&tma_bar[1], 1);
        mbar_fence_init();
    }
    pdl_wait();     // the previous kernel of the stream is done (the summary pass, a previous chunk's call)
    pdl_release();
    __syncthreads();
    if (kTma) {
        // (a.withhold: test only, a copy left out so that the wait for it runs out)
        const bool withheld = a.withhold && blockIdx.x == 0 && blockIdx.y == 0;
        if (tid == 0 && !withheld) p16_tma_chunk<NS, LPC>(maps, sm, &tma_bar[0], 0, row0, brow0, t_begin, has_z);
    } else {
        p16_issue_chunk<NS, LPC>(a, sm, 0, b, ch0, t_begin, has_z);
    }

    P16Consts<NSL> cc;
    bool small_a = false;  // some state with |A| < kZohFastMinA (0 included): the exact form
#pragma unroll
    for (int p = 0; p < NSL / 2; ++p) {
        float al[2], ni[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int n = e * NSL + 2 * p + q;
            const bool real = active && n < a.N;
            const float av = real ? __ldg(a.A + (size_t)d * a.N + n) : 0.0f;
            al[q] = av * kLog2e;
            ni[q] = av != 0.0f ? -1.0f / av : 0.0f;
            small_a |= real && !(fabsf(av) >= kZohFastMinA);
        }
        cc.al2[p] = pack2(al[0], al[1]);
        cc.ninv[p] = pack2(ni[0], ni[1]);
    }
    float w[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    float cb = 0.0f;
    if (kConv && active) {
        const int W = a.conv_width;
        const float* cw = a.conv_w + (size_t)d * W;
        // tap i of the 4-wide window is tap i - (4 - W) of the filter
        w[0] = W >= 4 ? __ldg(cw + 0 - (4 - W)) : 0.0f;
        w[1] = W >= 3 ? __ldg(cw + 1 - (4 - W)) : 0.0f;
        w[2] = W >= 2 ? __ldg(cw + 2 - (4 - W)) : 0.0f;
        w[3] = __ldg(cw + 3 - (4 - W));
        if (a.conv_b != nullptr) cb = __ldg(a.conv_b + d);
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] *= 0.5f;  // exact: the conv output enters SiLU as halves
        cb *= 0.5f;
    }
    const float dskip = (a.Dskip != nullptr && active) ? __ldg(a.Dskip + d) : 0.0f;
    const float bias = (a.delta_bias != nullptr && active) ? __ldg(a.delta_bias + d) : 0.0f;

    // this lane's states are n0 + i, i < NSL
    const int n0 = e * NSL;
    float h[NSL];
#pragma unroll
    for (int i = 0; i < NSL; ++i) h[i] = 0.0f;
    float dsum = 0.0f;
    if (kFinal) {
        // the state at the segment's start: h0 (its copy when the summaries ran first), or with a first
        // segment the end state of segment 0 from the first launch; then the later summaries folded in
        int s_first = 0;
        if (kSeg0 && seg > 0) {
            if (active) {
#pragma unroll
                for (int i = 0; i < NSL; ++i)
                    if (n0 + i < a.N) h[i] = a.ws_h[row * a.N + n0 + i];
            }
            s_first = 1;
        } else {
            const float* h0 = (!kSeg0 && a.nseg > 1) ? a.ws_h0 : a.h0;
            if (h0 != nullptr && active) {
#pragma unroll
                for (int i = 0; i < NSL; ++i)
                    if (n0 + i < a.N) h[i] = h0[row * a.N + n0 + i];
            }
        }
        for (int s = s_first; s < seg; ++s) {
            const float S = active ? a.ws_dsum[(size_t)s * rows + row] : 0.0f;
#pragma unroll
            for (int i = 0; i < NSL; ++i) {
                float al0, al1;
                unpack2(cc.al2[i / 2], al0, al1);
                const float hs = (active && n0 + i < a.N) ? a.ws_h[((size_t)s * rows + row) * a.N + n0 + i] : 0.0f;
                h[i] = fmaf(ex2((i & 1 ? al1 : al0) * S), h[i], hs);
            }
        }
    } else if (seg == 0 && a.ws_h0 != nullptr && a.h0 != nullptr && active) {
#pragma unroll
        for (int i = 0; i < NSL; ++i)
            if (n0 + i < a.N) a.ws_h0[row * a.N + n0 + i] = a.h0[row * a.N + n0 + i];
    }
    f32x2 hp[NSL / 2];
#pragma unroll
    for (int p = 0; p < NSL / 2; ++p) hp[p] = pack2(h[2 * p], h[2 * p + 1]);

    const bool exact = kZOH && __syncthreads_or(small_a);  // block-uniform choice of loop body
    const size_t yoff = row * (size_t)a.L;
    // the fast form takes its step in base-2 units (see p16_group): A unscaled, the bias times log2 e
    float bias_used = bias;
    if (kZOH && !exact) {
        bias_used = bias * kLog2e;
#pragma unroll
        for (int p = 0; p < NSL / 2; ++p) {
            float av[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int n = e * NSL + 2 * p + q;
                av[q] = (active && n < a.N) ? __ldg(a.A + (size_t)d * a.N + n) : 0.0f;
            }
            cc.al2[p] = pack2(av[0], av[1]);
        }
    }

    int buf = 0, k = 0;
    for (int c0 = t_begin; c0 < t_end; c0 += kP16Chunk, buf ^= 1, ++k) {
        if (kTma) {
            // the chunk's copies have landed (bounded wait; a block that gives up writes nothing more)
            const bool ok = mbar_wait_bounded(&tma_bar[buf], (unsigned)((k >> 1) & 1));
            if (__syncthreads_or(!ok)) {
                if (tid == 0) {
                    atomicOr(&g_scan_wait_error, 1u);
                    mbar_wait_bounded(&tma_bar[buf], (unsigned)((k >> 1) & 1));
                }
                return;
            }
            // every thread is done with the other buffers: refill them with the next chunk
            if (tid == 0 && c0 + kP16Chunk < t_end)
                p16_tma_chunk<NS, LPC>(maps, sm, &tma_bar[buf ^ 1], buf ^ 1, row0, brow0, c0 + kP16Chunk, has_z);
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            __syncthreads();  // chunk c0 landed for every thread; everyone is done with the other buffers
            if (c0 + kP16Chunk < t_end) p16_issue_chunk<NS, LPC>(a, sm, buf ^ 1, b, ch0, c0 + kP16Chunk, has_z);
        }
        if (kConv && c0 == 0 && a.conv_init != nullptr) {
            // x before t = 0 is the caller's history (oldest first), not the zeros the copy filled in
            const int W1 = a.conv_width - 1;
            for (int i = tid; i < kCh * W1; i += kP16Threads) {
                const int r = i / W1, k = i - r * W1;
                if (ch0 + r < a.D)
                    sm.x[buf][r][kP16Halo - W1 + k] =
                        static_cast<const uint16_t*>(a.conv_init)[((size_t)b * a.D + ch0 + r) * W1 + k];
            }
        }
        // widen B / C of this chunk to fp32 (consecutive threads write consecutive floats)
        for (int i = tid; i < 2 * NS * kP16Chunk; i += kP16Threads) {
            const int t = i / (2 * NS);
            const int rem = i - t * 2 * NS;
            const int wv = rem / NS, n = rem - wv * NS;
            sm.bc[t][wv][n] = n < a.N ? bf16_to_f32(sm.bcr[buf][wv][n][kBcOff + t]) : 0.0f;
        }
        __syncthreads();
        const int clen = min(kP16Chunk, t_end - c0);
        // every lane of a warp takes part (the shuffles need them); inactive channels write nothing
        for (int j0 = 0; j0 < clen; j0 += 8) {
            // h_all: every step; checkpoints: every 8th (c0 is a multiple of 8)
            const int hev = a.hall_every <= 1 ? 1 : 8;
            const int hsteps = (a.L + hev - 1) / hev;
            float* hall = kHall ? a.h_all + ((size_t)b * hsteps * a.D + (active ? d : 0)) * a.N + e * NSL +
                                          (size_t)(c0 / hev) * a.D * a.N
                                : nullptr;
            if (exact)
                p16_group<NS, LPC, Disc::kZOHExact, kFinal, kConv, kHall>(a, sm, buf, j0, cc, w, cb, dskip, bias, hp, dsum,
                                                                          has_z, active, yoff + c0, hall);
            else
                p16_group<NS, LPC, kZOH ? Disc::kZOH : Disc::kSimple, kFinal, kConv, kHall>(
                    a, sm, buf, j0, cc, w, cb, dskip, bias_used, hp, dsum, has_z, active, yoff + c0, hall);
        }
    }

    if (!active) return;
#pragma unroll
    for (int p = 0; p < NSL / 2; ++p) unpack2(hp[p], h[2 * p], h[2 * p + 1]);
    if (kFinal) {
        if (seg == a.nseg - 1 && a.h_out != nullptr) {
#pragma unroll
            for (int i = 0; i < NSL; ++i)
                if (n0 + i < a.N) a.h_out[row * a.N + n0 + i] = h[i];
        }
        if (kSeg0 && seg == 0) {  // the first carry of the L split
#pragma unroll
            for (int i = 0; i < NSL; ++i)
                if (n0 + i < a.N) a.ws_h[row * a.N + n0 + i] = h[i];
        }
    } else {
        if (e == 0) a.ws_dsum[(size_t)seg * rows + row] = dsum;
#pragma unroll
        for (int i = 0; i < NSL; ++i)
            if (n0 + i < a.N) a.ws_h[((size_t)seg * rows + row) * a.N + n0 + i] = h[i];
    }
}

template <int NS, int LPC, bool kZOH, bool kFinal, bool kConv, bool kHall = false, bool kTma = false,
          bool kSeg0 = false>
__global__ void __launch_bounds__(kP16Threads, p16_min_blocks(LPC))
    scan_p16_kernel(const ScanKernelArgs a, const __grid_constant__ P16Maps maps) {
    // with a first segment (kSeg0) the first launch has run segment 0's final pass: this final pass covers
    // segments 1 .. nseg - 1
    p16_run<NS, LPC, kZOH, kFinal, kConv, kHall, kTma, kSeg0>(a, maps, (int)blockIdx.z + ((kFinal && kSeg0) ? 1 : 0));
}

// The first launch of an L split with a first segment: block z = 0 runs segment 0's final pass (from h0;
// its end state becomes the first carry, and it needs no summary), blocks z >= 1 the summaries of
// segments 1 .. nseg - 2, at the same time.
template <int NS, int LPC, bool kZOH, bool kConv, bool kHall, bool kTma>
__global__ void __launch_bounds__(kP16Threads, p16_min_blocks(LPC))
    scan_p16_first_kernel(const ScanKernelArgs a, const __grid_constant__ P16Maps maps) {
    if (blockIdx.z == 0)
        p16_run<NS, LPC, kZOH, true, kConv, kHall, kTma, true>(a, maps, 0);
    else
        p16_run<NS, LPC, kZOH, false, kConv, false, kTma, true>(a, maps, (int)blockIdx.z);
}

// SSM_SCAN_STAGING=cpasync stages chunks with per-thread cp.async copies instead of the tiled bulk copies
// (for comparisons); the bulk copies are also skipped when a tensor map cannot be encoded.
inline bool p16_use_tma() {
    static const bool on = [] {
        const char* v = std::getenv("SSM_SCAN_STAGING");
        return !(v != nullptr && std::strcmp(v, "cpasync") == 0);
    }();
    return on;
}

template <int NS, int LPC>
inline bool p16_encode_maps(const ScanKernelArgs& a, P16Maps& m) {
    constexpr int kCh = P16Smem<NS, LPC>::kCh;
    const uint64_t L = (uint64_t)a.L, rows = (uint64_t)a.Bsz * a.D, brows = (uint64_t)a.Bsz * a.N;
    bool ok = encode_bf16_map_2d(&m.x, a.u, L, rows, L * 2, kP16Row, kCh) &&
              encode_bf16_map_2d(&m.dl, a.delta, L, rows, L * 2, kP16Row, kCh) &&
              encode_bf16_map_2d(&m.B, a.Bm, L, brows, L * 2, kP16Row, NS) &&
              encode_bf16_map_2d(&m.C, a.Cm, L, brows, L * 2, kP16Row, NS);
    if (ok && a.z != nullptr) ok = encode_bf16_map_2d(&m.zz, a.z, L, rows, L * 2, kP16Row, kCh);
    if (ok && a.z == nullptr) m.zz = m.x;  // never read: the z copy is skipped
    return ok;
}

template <int NS, int LPC, bool kZOH, bool kConv, bool kTma>
cudaError_t launch_p16_staged(const ScanKernelArgs& a, const P16Maps& maps, cudaStream_t stream) {
    const size_t smem = sizeof(P16Smem<NS, LPC>);
    constexpr int kCh = P16Smem<NS, LPC>::kCh;
    dim3 block(kP16Threads);
    const unsigned gx = (unsigned)((a.D + kCh - 1) / kCh);
    cudaError_t e;
    if (a.nseg > 1) {
        // the summaries of segments 0 .. nseg - 2, or with a first segment segment 0's final pass and the
        // summaries of segments 1 .. nseg - 2
        auto kfn = a.seg0_len > 0 ? (a.h_all != nullptr ? scan_p16_first_kernel<NS, LPC, kZOH, kConv, true, kTma>
                                                        : scan_p16_first_kernel<NS, LPC, kZOH, kConv, false, kTma>)
                                  : scan_p16_kernel<NS, LPC, kZOH, false, kConv, false, kTma>;
        e = set_dynamic_smem_once(kfn, (int)smem);
        if (e != cudaSuccess) return e;
        e = launch_pdl(kfn, dim3(gx, (unsigned)a.Bsz, (unsigned)(a.nseg - 1)), block, smem, stream, a, maps);
        if (e != cudaSuccess) return e;
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    auto kfn = a.seg0_len > 0 ? (a.h_all != nullptr ? scan_p16_kernel<NS, LPC, kZOH, true, kConv, true, kTma, true>
                                                    : scan_p16_kernel<NS, LPC, kZOH, true, kConv, false, kTma, true>)
                              : (a.h_all != nullptr ? scan_p16_kernel<NS, LPC, kZOH, true, kConv, true, kTma>
                                                    : scan_p16_kernel<NS, LPC, kZOH, true, kConv, false, kTma>);
    e = set_dynamic_smem_once(kfn, (int)smem);
    if (e != cudaSuccess) return e;
    ScanKernelArgs fa = a;
    fa.withhold = (kTma && a.nseg == 1 && withhold_first_copy()) ? 1 : 0;
    const unsigned gz = (unsigned)(a.seg0_len > 0 ? a.nseg - 1 : a.nseg);
    e = launch_pdl(kfn, dim3(gx, (unsigned)a.Bsz, gz), block, smem, stream, fa, maps);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int NS, int LPC, bool kZOH, bool kConv>
cudaError_t launch_p16_ns(const ScanKernelArgs& a, cudaStream_t stream) {
    P16Maps maps{};
    if (p16_use_tma() && p16_encode_maps<NS, LPC>(a, maps))
        return launch_p16_staged<NS, LPC, kZOH, kConv, true>(a, maps, stream);
    return launch_p16_staged<NS, LPC, kZOH, kConv, false>(a, maps, stream);
}

template <int NS, int LPC>
cudaError_t launch_p16(const ScanKernelArgs& a, int zoh, cudaStream_t s) {
    const bool conv = a.conv_w != nullptr;
    if (zoh) return conv ? launch_p16_ns<NS, LPC, true, true>(a, s) : launch_p16_ns<NS, LPC, true, false>(a, s);
    return conv ? launch_p16_ns<NS, LPC, false, true>(a, s) : launch_p16_ns<NS, LPC, false, false>(a, s);
}

}  // namespace ssm
