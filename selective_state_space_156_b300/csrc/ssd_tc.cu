// Mamba-2 (SSD) scan on the tcgen05 tensor cores: the chunked matrix ("dual") form of the selective
// recurrence with one scalar A per head (dpshk.com/news/3333417 section 6.1; pwwt.cn/news/5168881
// section 2.3: the semiseparable matrix splits into blocks that are processed like attention tiles).
//
// One CTA owns one (batch row b, head h) and walks its sequence in chunks of Q = 128 steps, carrying the
// state S (N x P, fp32, in registers: row n of S belongs to the threads of TMEM lane n).  With
// a_t = exp(dt_t A) and s_i = sum_{t0 <= j <= i} dt_j A (log2 units in the code), per chunk:
//
//   [G | C S]  = C [B ; S^T]^T                    (Q x (Q + P) over the N states)        tensor cores
//   M          = G o [j <= i] exp(s_i - s_j) w_j  + Dskip I                              threads -> TMEM
//   Y          = exp(s_i) (C S) + M X              (inter-chunk + intra-chunk + skip)    tensor cores
//   S         <- exp(s_end) S + B^T (v o X)^T,    v_j = exp(s_end - s_j) w_j             tensor cores
//   y          = Y * SiLU(z)
//
// where w_j = dt_j (simplified input scale) or expm1(dt_j A) / A (zero-order hold).  C, B (Q x N) and X
// (the head's P channels over the chunk) arrive by TMA in the 128-byte swizzle layout; the increment reads
// B as it landed, as an MN-major operand.  The operands the threads build (M, v o X, S^T) carry two bf16
// terms, hi = bf16(u) and lo = bf16(u - hi), and every product with them is issued for both terms into
// one accumulator, so their rounding costs about 2^-16 relative instead of 2^-8.  v o X and S^T are
// written to shared memory in the copies' layout; S^T's two terms sit right below B in the same K blocks
// (one N = 128 product per K step for each of G and C S).  M goes back into tensor memory over the G block
// it was built from (16 fp32 columns of G hold the 8 + 8 columns of M's two terms) and is the A operand
// of M X from there: it never passes through shared memory.
//
// Accumulators in TMEM: G (then M) in columns 0..127, C S_hi in 128..191, C S_lo in 192..255, M X in
// 256..319 and the state increment in 320..383.  A dedicated warp issues the copies and the products; four compute
// warpgroups split the element-wise work (each warp reads the TMEM lanes of its quarter of the rows).
// Overlaps within a chunk: G is issued first and completes on its own, so that the M build starts while
// C S is still on the tensor cores; the increment is issued as soon as v o X is built and runs while the
// threads build M; it completes on a barrier of its own, so that the state update runs while M X is still
// on the tensor cores.  Across chunks: the next chunk's C is fetched as soon as this chunk's C S is done,
// its B, X and dt as soon as M X and the increment are; y leaves through a TMA store of a staged
// tile.  Every product's shared-memory descriptors are built once; a K step adds a constant.
#include <cstdint>

#include "bulk_copy.cuh"
#include "ssm_device.cuh"
#include "ssm_internal.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace ssm {

namespace {

constexpr int kQ = 128;   // chunk length
constexpr int kN = 128;   // state size of the tiles; a problem with N = 64 leaves states 64..127 zero
constexpr int kP = 64;    // channels per head
#ifndef SSD_COMPUTE_WARPGROUPS
#define SSD_COMPUTE_WARPGROUPS 4
#endif
constexpr int kWG = SSD_COMPUTE_WARPGROUPS;  // compute warpgroups
constexpr int kCompute = 128 * kWG;          // compute threads
constexpr int kIssuer = 4 * kWG;             // the warp that issues copies and products
constexpr int kThreads = kCompute + 32;

// Shared memory, from a 1024-byte-aligned base.  Tiles are 128-byte swizzled in K blocks of 64 elements;
// swz() gives the byte offset of (row, k) for a K-block stride.
constexpr int kOffC = 0;                         // C: Q rows (t) x N, K blocks of 16 KB
constexpr int kBS = 32768;                       // K-block stride of the [B ; S^T hi ; S^T lo] operand:
constexpr int kOffBS = kOffC + 2 * 16384;        //   rows 0..127 B (t x n), 128..191 S^T hi and 192..255
constexpr int kRowStHi = 128, kRowStLo = 192;    //   S^T lo (p x n)
constexpr int kOffX = kOffBS + 2 * kBS;          // X: P rows (p) x Q (t), K blocks of 8 KB
constexpr int kOffXs = kOffX + 2 * 8192;         // v o X hi, the same shape
constexpr int kOffXsLo = kOffXs + 2 * 8192;      // v o X lo
constexpr int kOffY = kOffXsLo + 2 * 8192;       // the y tile: P rows (p) x Q (t), K blocks of 8 KB
constexpr int kOffS2 = kOffY + 2 * 8192;         // float s[Q]: cumulative log2 decay
constexpr int kOffW = kOffS2 + kQ * 4;           // float w[Q]: input scale
constexpr int kOffV = kOffW + kQ * 4;            // float v[Q]: exp2(s_end - s_j) w_j
constexpr int kOffWarp = kOffV + kQ * 4;         // float[4]: warp totals of the prefix sum
constexpr int kOffDt = kOffWarp + 16;            // bf16 dt[Q] of the chunk, copied with B and X
constexpr int kOffBar = kOffDt + kQ * 2;         // uint64 barriers: C landed, B and X landed, products
                                                 //   done, increment done, C S done
constexpr int kOffTmem = kOffBar + 48;           // uint32 TMEM base, int abort flag
constexpr int kSmemUsed = kOffTmem + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;     // slack for aligning the base
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColG = 0, kColY1 = 128, kColY2 = 256, kColSc = 320;
constexpr unsigned kCBytes = kQ * kN * 2, kBBytes = kQ * kN * 2, kXBytes = kP * kQ * 2;   // per chunk

__device__ unsigned int g_ssd_wait_error = 0;

__host__ __device__ constexpr uint32_t swz(int kb_stride, int row, int k) {
    return static_cast<uint32_t>((k >> 6) * kb_stride + row * 128 + ((((k >> 3) & 7) ^ (row & 7)) << 4) +
                                 ((k & 7) << 1));
}

// the compute threads alone (the issuer warp does not take part)
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, %0;" ::"r"(kCompute) : "memory"); }

// This thread waits for the phase; false when it gave up (about one second) or some thread of the block
// already had, in which case it raises, or finds, the block's abort flag.  After an abort the block runs
// its loop to the end without waiting or issuing anything, so that every thread still meets every
// barrier, and reports the failure.
__device__ __forceinline__ bool wait_own(uint64_t* bar, unsigned parity, volatile int* abort_flag) {
    if (*abort_flag) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void st_shared_v4(unsigned char* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(p)), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_shared_u32(unsigned char* p, uint32_t a) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(a) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(const unsigned char* p) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

// two floats as a bf16x2 hi word and the bf16x2 word of what hi leaves over
__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16x2(a, b);
    lo = pack_bf16x2(a - bf16_lo(hi), b - bf16_hi(hi));
}

// Lanes r and r ^ 1 hold the same columns of rows r and r ^ 1 of a row-per-lane matrix; the transposed
// tile wants (column, row pair) words.  For the column pair (c, c + 1) the even lane returns the pair of
// rows (r, r + 1) of column c, the odd lane that of column c + 1, and `col` tells which.
__device__ __forceinline__ void pair_rows(float own_c, float own_c1, int odd, float& first, float& second) {
    const float recv = __shfl_xor_sync(0xffffffffu, odd ? own_c : own_c1, 1);
    first = odd ? recv : own_c;
    second = odd ? own_c1 : recv;
}

__global__ void __launch_bounds__(kThreads, 1)
    ssd_chunk_kernel(const SsdArgs a, const __grid_constant__ CUtensorMap map_c, const __grid_constant__ CUtensorMap map_b,
                     const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_y) {
    constexpr int kPW = kP / kWG;   // channels p whose outputs and state each compute warpgroup owns
    static_assert(kPW % 16 == 0, "warpgroup split");
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    unsigned char* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool issuer_warp = warp == kIssuer;
    const bool issuer = issuer_warp && lane == 0;
    const int r = tid & 127;        // compute threads: TMEM lane, step i of the chunk, state n
    const int wg = tid >> 7;        // compute warpgroup (kWG for the issuer warp)
    const int odd = r & 1;
    const int b = blockIdx.x / a.H, h = blockIdx.x % a.H;
    const int bg = b * a.G + h / (a.H / a.G);
    const int L = a.L;
    const size_t row0 = (static_cast<size_t>(b) * a.H + h) * kP;   // first channel row of this head in (B*D, L)
    const size_t dt_row = (static_cast<size_t>(b) * a.H + h) * L;

    uint64_t* bar_c = reinterpret_cast<uint64_t*>(sm + kOffBar);
    uint64_t* bar_bx = bar_c + 1;
    uint64_t* mma_bar = bar_c + 2;
    uint64_t* inc_bar = bar_c + 3;   // the chunk's state increment is done
    uint64_t* cs_bar = bar_c + 4;    // the chunk's C S is done (C may be overwritten)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffTmem);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kOffTmem + 4);
    float* s2s = reinterpret_cast<float*>(sm + kOffS2);
    float* wsv = reinterpret_cast<float*>(sm + kOffW);
    float* vsv = reinterpret_cast<float*>(sm + kOffV);
    float* wsum = reinterpret_cast<float*>(sm + kOffWarp);

    auto issue_c = [&](int cc) {
        mbar_arrive_expect_tx(bar_c, kCBytes);
        tma_load_3d(sm + kOffC, &map_c, 0, cc * kQ, bg, bar_c);
        tma_load_3d(sm + kOffC + 16384, &map_c, 64, cc * kQ, bg, bar_c);
    };
    auto issue_bx = [&](int cc) {
        const unsigned dt_bytes = static_cast<unsigned>(min(kQ, L - cc * kQ)) * 2u;   // L % 8 == 0: whole 16 B
        mbar_arrive_expect_tx(bar_bx, kBBytes + kXBytes + dt_bytes);
        bulk_g2s(sm + kOffDt, reinterpret_cast<const uint16_t*>(a.dt) + dt_row + cc * kQ, dt_bytes, bar_bx);
        tma_load_3d(sm + kOffBS, &map_b, 0, cc * kQ, bg, bar_bx);
        tma_load_3d(sm + kOffBS + kBS, &map_b, 64, cc * kQ, bg, bar_bx);
        tma_load_2d(sm + kOffX, &map_x, cc * kQ, static_cast<int>(row0), bar_bx);
        tma_load_2d(sm + kOffX + 8192, &map_x, cc * kQ + 64, static_cast<int>(row0), bar_bx);
    };

    bool c_pend_init = true;
    if (issuer) {
        *abort_flag = 0;
        mbar_init(bar_c, 1);
        mbar_init(bar_bx, 1);
        mbar_init(mma_bar, 1);
        mbar_init(inc_bar, 1);
        mbar_init(cs_bar, 1);
        mbar_fence_init();
        tma_prefetch_map(&map_c);
        tma_prefetch_map(&map_b);
        tma_prefetch_map(&map_x);
        tma_prefetch_map(&map_y);
        if (a.withhold)
            c_pend_init = false;   // test only: chunk 0's C is never copied, so every wait for it runs out
        else
            issue_c(0);
        issue_bx(0);
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }

    const float A = a.A[h];
    const float A2 = A * kLog2e;
    const float bias = a.dt_bias ? a.dt_bias[h] : 0.0f;
    const float dsk = a.Dskip ? a.Dskip[h] : 0.0f;

    // compute threads: their part of the state, S[n = r][p] for the warpgroup's channels, and S^T (hi, lo)
    float S[kPW];
    if (!issuer_warp) {
#pragma unroll
        for (int q = 0; q < kPW; q += 2) {
            const int p = wg * kPW + q;
            S[q] = (a.h0 && r < a.N) ? a.h0[(row0 + p) * a.N + r] : 0.0f;
            S[q + 1] = (a.h0 && r < a.N) ? a.h0[(row0 + p + 1) * a.N + r] : 0.0f;
            float f, s;
            pair_rows(S[q], S[q + 1], odd, f, s);
            uint32_t hi, lo;
            split_pair(f, s, hi, lo);
            st_shared_u32(sm + kOffBS + swz(kBS, kRowStHi + p + odd, r & ~1), hi);
            st_shared_u32(sm + kOffBS + swz(kBS, kRowStLo + p + odd, r & ~1), lo);
        }
    }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = static_cast<uint32_t>((warp & 3) * 32) << 16;   // this warp's TMEM lanes

    const uint32_t sC = smem_u32(sm + kOffC), sBS = smem_u32(sm + kOffBS), sX = smem_u32(sm + kOffX);
    const uint32_t sXs = smem_u32(sm + kOffXs), sXsLo = smem_u32(sm + kOffXsLo);

    // the operands' shared-memory descriptors, built once: a K step only moves the start address, which is
    // the descriptor's low field (address / 16), so each product adds a constant to a base descriptor
    const uint64_t dC = tc::desc_k_sw128(sC), dBS = tc::desc_k_sw128(sBS), dX = tc::desc_k_sw128(sX);
    const uint64_t dXs = tc::desc_k_sw128(sXs), dXsLo = tc::desc_k_sw128(sXsLo);
    const uint64_t dBmn = tc::desc_mn_sw128(sBS, kBS, 1024);

    unsigned c_phase = 0, bx_phase = 0, mma_phase = 0;
    // the issuer's view of its asynchronous work: issued and not yet seen complete by its own wait, with
    // the parity of the phase that completes it (a chunk's copies: the chunk's; products: their order)
    // one bit per barrier (C, B X, products, increment, C S) in `pend`, and the awaited parity in `par`
    enum : unsigned { kPC = 1u, kPBX = 2u, kPMMA = 4u, kPINC = 8u, kPCS = 16u };
    unsigned pend = (c_pend_init ? kPC : 0u) | kPBX, par = 0u;
    auto set_pend = [&](unsigned bit, unsigned parity) { pend |= bit; par = parity ? (par | bit) : (par & ~bit); };
    const int nchunks = (L + kQ - 1) / kQ;
    for (int c = 0; c < nchunks; ++c) {
        const int t0 = c * kQ;
        // this chunk's C, B, X and dt (issued a phase ahead); each thread waits for itself
        if (wait_own(bar_c, c_phase, abort_flag)) pend &= ~kPC;
        if (wait_own(bar_bx, bx_phase, abort_flag)) pend &= ~kPBX;
        c_phase ^= 1u;
        bx_phase ^= 1u;

        float s2_end = 0.0f, s2_row = 0.0f;
        if (issuer && !*abort_flag) {
            // G = C B^T first (the M build waits for it alone), then [C S_hi | C S_lo] = C [S^T hi ; S^T lo]^T,
            // which runs under the M build: eight N = 128 products each
            tc::fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t ka = (ks >> 2) * 16384 + (ks & 3) * 32;
                const uint32_t kb = (ks >> 2) * kBS + (ks & 3) * 32;
                tc::mma_bf16(tmem + kColG, dC + (ka >> 4), dBS + (kb >> 4), tc::idesc_bf16(128, 128), ks > 0);
            }
            tc::mma_commit(mma_bar);
            set_pend(kPMMA, 0u);   // the first of the chunk's two commits
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t ka = (ks >> 2) * 16384 + (ks & 3) * 32;
                const uint32_t kb = (ks >> 2) * kBS + kRowStHi * 128 + (ks & 3) * 32;
                tc::mma_bf16(tmem + kColY1, dC + (ka >> 4), dBS + (kb >> 4), tc::idesc_bf16(128, 128), ks > 0);
            }
            tc::mma_commit(cs_bar);
            set_pend(kPCS, c & 1);
        }
        if (issuer) {
            bulk_wait_read_all();   // the previous chunk's y store has left the y tile (before its next writes)
        } else if (!issuer_warp) {
            // meanwhile: step sizes and the cumulative decay of the chunk, by warpgroup 0 (steps past L:
            // dt = 0, so a = 1 and w = 0)
            float inc = 0.0f;
            if (wg == 0) {
                float dtv = 0.0f;
                if (t0 + r < L) {
                    const float sr = bf16_to_f32(reinterpret_cast<const uint16_t*>(sm + kOffDt)[r]) + bias;
                    dtv = a.softplus ? softplus_fast(sr) : sr;
                }
                inc = dtv * A2;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float u = __shfl_up_sync(0xffffffffu, inc, o);
                    if (lane >= o) inc += u;
                }
                if (lane == 31) wsum[warp] = inc;
                wsv[r] = (a.zoh && A != 0.0f) ? expm1f(dtv * A) / A : dtv;
            }
            compute_sync();
            if (wg == 0) {
                for (int w2 = 0; w2 < warp; ++w2) inc += wsum[w2];
                s2s[r] = inc;
            }
            compute_sync();
            s2_end = s2s[kQ - 1];
            s2_row = s2s[r];
            if (wg == 0) vsv[r] = ex2(s2_end - s2_row) * wsv[r];
            compute_sync();
            // v o X (hi, lo) in 16-byte pieces of 8 steps, dealt over the compute threads
#pragma unroll 1
            for (int idx = tid; idx < kP * (kQ / 8); idx += kCompute) {
                const int p = idx >> 4, tc8 = (idx & 15) * 8;
                const uint32_t o = swz(8192, p, tc8);
                const uint4 xv = ld_shared_v4(sm + kOffX + o);
                const float4 v0 = *reinterpret_cast<const float4*>(vsv + tc8);
                const float4 v1 = *reinterpret_cast<const float4*>(vsv + tc8 + 4);
                uint32_t hi[4], lo[4];
                split_pair(bf16_lo(xv.x) * v0.x, bf16_hi(xv.x) * v0.y, hi[0], lo[0]);
                split_pair(bf16_lo(xv.y) * v0.z, bf16_hi(xv.y) * v0.w, hi[1], lo[1]);
                split_pair(bf16_lo(xv.z) * v1.x, bf16_hi(xv.z) * v1.y, hi[2], lo[2]);
                split_pair(bf16_lo(xv.w) * v1.z, bf16_hi(xv.w) * v1.w, hi[3], lo[3]);
                st_shared_v4(sm + kOffXs + o, hi[0], hi[1], hi[2], hi[3]);
                st_shared_v4(sm + kOffXsLo + o, lo[0], lo[1], lo[2], lo[3]);
            }
            tc::fence_async_smem();   // v o X, read by the increment issued after the next barrier
        }
        if (wait_own(mma_bar, mma_phase, abort_flag) && issuer) pend &= ~kPMMA;
        mma_phase ^= 1u;
        tc::fence_before();
        __syncthreads();   // v o X is complete (and G is read by the M build behind this)
        tc::fence_after();
        if (issuer && !*abort_flag) {
            // the increment B^T (v o X)^T (both terms of v o X), B read MN-major, under the M build
#pragma unroll
            for (int ks = 0; ks < 16; ++ks) {
                const int k = ks & 7;
                const uint32_t ka = k * 2048;   // 16 steps (rows t) of B per K step
                const uint32_t kb = (k >> 2) * 8192 + (k & 3) * 32;
                tc::mma_bf16(tmem + kColSc, dBmn + (ka >> 4), (ks < 8 ? dXs : dXsLo) + (kb >> 4),
                             tc::idesc_bf16(128, kP, true), ks > 0);
            }
            tc::mma_commit(inc_bar);
            set_pend(kPINC, c & 1);
            // C is free once C S is done: the next chunk's copy overlaps the rest of this one
            if (wait_own(cs_bar, c & 1, abort_flag)) pend &= ~kPCS;
            if (c + 1 < nchunks && !*abort_flag) {
                issue_c(c + 1);
                set_pend(kPC, (c + 1) & 1);
            }
        }

        // row i = r of M from row i of G, in 16-column blocks dealt round-robin to the warpgroups; blocks
        // wholly above the diagonal are zeros
        if (!issuer_warp) {
            const int quarter = warp & 3;
            const f32x2 srow2 = pack2(s2_row, s2_row);
#pragma unroll 1
            for (int cb = wg; cb < kQ / 16; cb += kWG) {
                const int jb = cb * 16;
                float gv[16];
                const bool live = 32 * quarter + 31 >= jb;   // warp-uniform: some row of this warp reaches jb
                if (live) tc::tmem_ld16(tmem + tlane + kColG + jb, gv);
                // the block's 16 columns of M as bf16 pairs: hi terms, then lo terms, written over the G block
                // just read (its 16 fp32 columns hold 8 columns of each), the A operand of M X
                uint32_t hi8[8], lo8[8];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t* hi = hi8 + 4 * q;
                    uint32_t* lo = lo8 + 4 * q;
#pragma unroll
                    for (int e = 0; e < 4; ++e) hi[e] = lo[e] = 0u;
                    const int j0 = jb + q * 8;
                    if (live && j0 <= r) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = j0 + 2 * e;
                            const float2 sj = *reinterpret_cast<const float2*>(s2s + j);
                            const float2 wj = *reinterpret_cast<const float2*>(wsv + j);
                            const f32x2 ex = ex2x2(sub2(srow2, pack2(sj.x, sj.y)));
                            const f32x2 m = mul2(mul2(pack2(gv[q * 8 + 2 * e], gv[q * 8 + 2 * e + 1]), ex),
                                                 pack2(wj.x, wj.y));
                            float v0, v1;
                            unpack2(m, v0, v1);
                            if (j0 + 8 > r) {   // the diagonal piece: mask above it, D skip on it
                                v0 = j < r ? v0 : (j == r ? dsk + v0 : 0.0f);
                                v1 = j + 1 < r ? v1 : (j + 1 == r ? dsk + v1 : 0.0f);
                            }
                            split_pair(v0, v1, hi[e], lo[e]);
                        }
                    }
                }
                tc::tmem_st8(tmem + tlane + kColG + jb, hi8);
                tc::tmem_st8(tmem + tlane + kColG + jb + 8, lo8);
            }
            tc::tmem_wait_st();
        }
        tc::fence_async_smem();   // v o X
        tc::fence_before();
        __syncthreads();

        if (issuer && !*abort_flag) {
            // M X (both terms of M, A from tensor memory); the commit also covers the increment issued before it
            tc::fence_after();
#pragma unroll
            for (int ks = 0; ks < 16; ++ks) {
                const int k = ks & 7;
                const uint32_t ta = tmem + kColG + 16 * k + (ks < 8 ? 0u : 8u);
                const uint32_t kb = (k >> 2) * 8192 + (k & 3) * 32;
                tc::mma_bf16_ts(tmem + kColY2, ta, dX + (kb >> 4), tc::idesc_bf16(128, kP), ks > 0);
            }
            tc::mma_commit(mma_bar);
            set_pend(kPMMA, 1u);   // the second
        }
        // the state first, while M X runs: S <- exp2(s_end) S + increment (row n = r), S^T (hi, lo) for the
        // next chunk
        if (wait_own(inc_bar, c & 1, abort_flag) && issuer) pend &= ~kPINC;
        tc::fence_after();
        if (!issuer_warp) {
            const float eend = ex2(s2_end);
#pragma unroll
            for (int pc = 0; pc < kPW / 16; ++pc) {
                const int pb = wg * kPW + pc * 16;
                float sc[16];
                tc::tmem_ld16(tmem + tlane + kColSc + pb, sc);
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    const int q = pc * 16 + e;
                    S[q] = fmaf(eend, S[q], sc[e]);
                    S[q + 1] = fmaf(eend, S[q + 1], sc[e + 1]);
                    float f, s2v;
                    pair_rows(S[q], S[q + 1], odd, f, s2v);
                    uint32_t hi, lo;
                    split_pair(f, s2v, hi, lo);
                    st_shared_u32(sm + kOffBS + swz(kBS, kRowStHi + pb + e + odd, r & ~1), hi);
                    st_shared_u32(sm + kOffBS + swz(kBS, kRowStLo + pb + e + odd, r & ~1), lo);
                }
            }
        }
        if (wait_own(mma_bar, mma_phase, abort_flag) && issuer) pend &= ~kPMMA;
        mma_phase ^= 1u;
        tc::fence_after();
        if (issuer && c + 1 < nchunks && !*abort_flag) {   // B and X are free
            issue_bx(c + 1);
            set_pend(kPBX, (c + 1) & 1);
        }

        if (!issuer_warp) {
            // outputs of row i = r (step t), this warpgroup's channels: C S (both terms) and M X from TMEM,
            // y staged as the y tile
            const int t = t0 + r;
            const float ei = ex2(s2_row);
#pragma unroll
            for (int pc = 0; pc < kPW / 16; ++pc) {
                const int pb = wg * kPW + pc * 16;
                float y1[16], v[2][16];
                {
                    const uint32_t ta[2] = {tmem + tlane + kColY1 + pb, tmem + tlane + kColY1 + kP + pb};
                    tc::tmem_ld16xn<2>(ta, v);
#pragma unroll
                    for (int e = 0; e < 16; ++e) y1[e] = v[0][e] + v[1][e];
                }
                tc::tmem_ld16(tmem + tlane + kColY2 + pb, v[0]);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    y1[e] = fmaf(ei, y1[e], v[0][e]);
                    if (a.z && t < L)
                        y1[e] *= silu(bf16_to_f32(reinterpret_cast<const uint16_t*>(a.z)[(row0 + pb + e) * L + t]));
                }
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    float f, s2v;
                    pair_rows(y1[e], y1[e + 1], odd, f, s2v);
                    st_shared_u32(sm + kOffY + swz(8192, pb + e + odd, r & ~1), pack_bf16x2(f, s2v));
                }
            }
        }
        tc::fence_async_smem();   // the y tile and S^T
        tc::fence_before();
        __syncthreads();          // every TMEM and shared read of this chunk is done
        if (issuer && !*abort_flag) {
            tma_store_2d(&map_y, t0, static_cast<int>(row0), sm + kOffY);
            if (t0 + 64 < L) tma_store_2d(&map_y, t0 + 64, static_cast<int>(row0), sm + kOffY + 8192);
            bulk_commit_group();
        }
    }

    const bool ok = *abort_flag == 0;   // read after the loop's last barrier: the same on every thread
    if (ok) {
        if (a.h_out && !issuer_warp) {
#pragma unroll
            for (int q = 0; q < kPW; ++q)
                if (r < a.N) a.h_out[(row0 + wg * kPW + q) * a.N + r] = S[q];
        }
    } else if (issuer) {
        // a wait gave up: record it and let this block's copies and products still in flight end (bounded;
        // products complete in order, so the last commit covers every earlier one)
        atomicOr(&g_ssd_wait_error, 1u);
        if (pend & kPC) mbar_wait_bounded(bar_c, (par & kPC) ? 1u : 0u);
        if (pend & kPBX) mbar_wait_bounded(bar_bx, (par & kPBX) ? 1u : 0u);
        if (pend & kPINC) mbar_wait_bounded(inc_bar, (par & kPINC) ? 1u : 0u);
        if (pend & kPCS) mbar_wait_bounded(cs_bar, (par & kPCS) ? 1u : 0u);
        if (pend & kPMMA) mbar_wait_bounded(mma_bar, (par & kPMMA) ? 1u : 0u);
    }
    if (issuer) bulk_wait_all();   // the y stores are complete
    tc::fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

// N = 64 runs the same tiles: the B and C maps end at state 64, so the copies fill states 64..127 with
// zeros, which leave G, C S and the increment exact and those rows of S at zero.
bool ssd_tc_supported(int N, int P) { return (N == kN || N == 64) && P == kP; }

cudaError_t launch_ssd_chunked(const SsdArgs& a, cudaStream_t stream) {
    CUtensorMap mc, mb, mx, my;
    const uint64_t bc_dims[3] = {static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.L),
                                 static_cast<uint64_t>(a.Bsz) * a.G};
    const uint64_t bc_strides[2] = {static_cast<uint64_t>(a.N) * 2, static_cast<uint64_t>(a.L) * a.N * 2};
    const uint32_t bc_box[3] = {64, kQ, 1};
    const uint64_t x_dims[2] = {static_cast<uint64_t>(a.L), static_cast<uint64_t>(a.Bsz) * a.H * kP};
    const uint64_t x_strides[1] = {static_cast<uint64_t>(a.L) * 2};
    const uint32_t x_box[2] = {64, kP};
    if (!encode_bf16_map_sw128(&mc, a.Cm, 3, bc_dims, bc_strides, bc_box) ||
        !encode_bf16_map_sw128(&mb, a.Bm, 3, bc_dims, bc_strides, bc_box) ||
        !encode_bf16_map_sw128(&mx, a.x, 2, x_dims, x_strides, x_box) ||
        !encode_bf16_map_sw128(&my, a.y, 2, x_dims, x_strides, x_box))
        return cudaErrorInvalidValue;
    cudaError_t e = set_dynamic_smem_once(ssd_chunk_kernel, kSmemBytes);
    if (e != cudaSuccess) return e;
    SsdArgs args = a;
    args.withhold = withhold_first_copy() ? 1 : 0;
    ssd_chunk_kernel<<<a.Bsz * a.H, kThreads, kSmemBytes, stream>>>(args, mc, mb, mx, my);
    return cudaGetLastError();
}

cudaError_t take_ssd_wait_error(unsigned* flags) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_ssd_wait_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_ssd_wait_error, &zero, sizeof(unsigned));
}

}  // namespace ssm
