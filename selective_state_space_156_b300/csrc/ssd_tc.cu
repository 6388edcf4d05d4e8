// Mamba-2 (SSD) scan on the tcgen05 tensor cores: the chunked matrix ("dual") form of the selective
// recurrence with one scalar A per head (dpshk.com/news/3333417 section 6.1; pwwt.cn/news/5168881
// section 2.3: the semiseparable matrix splits into blocks that are processed like attention tiles).
//
// One CTA owns one (batch row b, head h) and walks its sequence in chunks of Q = 128 steps, carrying the
// state S (N x P, fp32, in registers: thread n holds row n).  With a_t = exp(dt_t A) and
// s_i = sum_{t0 <= j <= i} dt_j A (log2 units in the code), per chunk:
//
//   G     = C B^T                                (Q x Q, over the N states)           tensor cores
//   M     = G o [j <= i] exp(s_i - s_j) w_j      (the decayed causal mask)            threads -> smem
//   Y     = exp(s_i) (C S) + M X                 (inter-chunk + intra-chunk)          tensor cores
//   S    <- exp(s_end) S + (exp(s_end - s_j) w_j B_j)^T X                              tensor cores
//   y     = (Y + Dskip x) * SiLU(z)
//
// where w_j = dt_j (simplified input scale) or expm1(dt_j A) / A (zero-order hold), C, B (Q x N) and X
// (the head's P channels over the chunk) arrive by TMA in the 128-byte swizzle layout, and the operands
// built by threads (M, the scaled B^T, S^T) are written in the same layout as hi + lo bf16 pairs.
// Accumulators live in TMEM: G in columns 0..127 (then the state increment in 0..63), C S in 128..191,
// M X in 192..255.
#include <cstdint>

#include "bulk_copy.cuh"
#include "ssm_device.cuh"
#include "ssm_internal.h"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace ssm {

namespace {

constexpr int kQ = 128;   // chunk length
constexpr int kN = 128;   // state size
constexpr int kP = 64;    // channels per head
constexpr int kThreads = 128;

// shared memory, from a 1024-byte-aligned base.  The operands built by threads are each stored as two
// bf16 terms, hi = bf16(v) and lo = bf16(v - hi), and every product with them is issued twice into the
// same accumulator: the rounding of those operands then costs about 2^-16 relative instead of 2^-8.
constexpr int kOffC = 0;                        // C chunk: Q rows (t) x N (n), two K blocks of 16 KB
constexpr int kOffB = kOffC + kQ * kN * 2;      // B chunk, the same shape; once G = C B^T and the scaled
constexpr int kOffMlo = kOffB;                  //   B^T are built, the lo term of M takes its place
constexpr int kOffX = kOffB + kQ * kN * 2;      // X chunk: P rows (p) x Q (t), two K blocks of 8 KB
constexpr int kOffM = kOffX + kP * kQ * 2;      // M (hi): Q rows (i) x Q (j)
constexpr int kOffBt = kOffM + kQ * kQ * 2;     // scaled B^T (hi): N rows (n) x Q (t)
constexpr int kOffBtLo = kOffBt + kN * kQ * 2;  // scaled B^T (lo)
constexpr int kOffSt = kOffBtLo + kN * kQ * 2;  // S^T (hi): P rows (p) x N (n)
constexpr int kOffStLo = kOffSt + kP * kN * 2;  // S^T (lo)
constexpr int kOffS2 = kOffStLo + kP * kN * 2;  // float s[Q]: cumulative log2 decay
constexpr int kOffW = kOffS2 + kQ * 4;          // float w[Q]: input scale
constexpr int kOffV = kOffW + kQ * 4;           // float v[Q]: exp2(s_end - s_j) w_j
constexpr int kOffWarp = kOffV + kQ * 4;        // float[4]: warp totals of the prefix sum
constexpr int kOffBar = kOffWarp + 16;          // uint64 tma barrier, mma barrier
constexpr int kOffTmem = kOffBar + 16;          // uint32 TMEM base
constexpr int kSmemUsed = kOffTmem + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;    // slack for aligning the base
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColG = 0, kColSc = 0, kColY1 = 128, kColY2 = 192;
constexpr unsigned kTileBytes = 2 * kQ * kN * 2 + kP * kQ * 2;   // C + B + X per chunk

__device__ unsigned int g_ssd_wait_error = 0;

// every thread waits; false on every thread if any of them gave up
__device__ __forceinline__ bool wait_all(uint64_t* bar, unsigned parity) {
    const bool ok = mbar_wait_bounded(bar, parity);
    return __syncthreads_or(!ok) == 0;
}

__device__ __forceinline__ void st_shared_v4(unsigned char* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(p)), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// two floats as a bf16x2 hi word and the bf16x2 word of what hi leaves over
__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16x2(a, b);
    lo = pack_bf16x2(a - bf16_lo(hi), b - bf16_hi(hi));
}

__device__ __forceinline__ float ld_bf16_shared(const unsigned char* p) {
    return bf16_to_f32(*reinterpret_cast<const uint16_t*>(p));
}

__global__ void __launch_bounds__(kThreads, 1)
    ssd_chunk_kernel(const SsdArgs a, const __grid_constant__ CUtensorMap map_c, const __grid_constant__ CUtensorMap map_b,
                     const __grid_constant__ CUtensorMap map_x) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    unsigned char* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x / a.H, h = blockIdx.x % a.H;
    const int g = h / (a.H / a.G);
    const int L = a.L;
    const size_t row0 = (static_cast<size_t>(b) * a.H + h) * kP;   // first channel row of this head in (B*D, L)

    uint64_t* tma_bar = reinterpret_cast<uint64_t*>(sm + kOffBar);
    uint64_t* mma_bar = tma_bar + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffTmem);
    float* s2s = reinterpret_cast<float*>(sm + kOffS2);
    float* wsv = reinterpret_cast<float*>(sm + kOffW);
    float* vsv = reinterpret_cast<float*>(sm + kOffV);
    float* wsum = reinterpret_cast<float*>(sm + kOffWarp);

    if (tid == 0) {
        mbar_init(tma_bar, 1);
        mbar_init(mma_bar, 1);
        mbar_fence_init();
        tma_prefetch_map(&map_c);
        tma_prefetch_map(&map_b);
        tma_prefetch_map(&map_x);
    }
    if (warp == 0) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = static_cast<uint32_t>(warp * 32) << 16;   // this warp's TMEM lanes

    const float A = a.A[h];
    const float A2 = A * kLog2e;
    const float bias = a.dt_bias ? a.dt_bias[h] : 0.0f;
    const float dsk = a.Dskip ? a.Dskip[h] : 0.0f;

    // the state, row n = tid of S (N x P)
    float S[kP];
#pragma unroll
    for (int p = 0; p < kP; ++p) S[p] = a.h0 ? a.h0[(row0 + p) * kN + tid] : 0.0f;

    const uint32_t sC = smem_u32(sm + kOffC), sB = smem_u32(sm + kOffB), sX = smem_u32(sm + kOffX);
    const uint32_t sM = smem_u32(sm + kOffM), sMlo = smem_u32(sm + kOffMlo);
    const uint32_t sBt = smem_u32(sm + kOffBt), sBtLo = smem_u32(sm + kOffBtLo);
    const uint32_t sSt = smem_u32(sm + kOffSt), sStLo = smem_u32(sm + kOffStLo);

    unsigned tma_phase = 0, mma_phase = 0;
    bool tma_pending = false, mma_pending = false, ok = true;
    const int nchunks = (L + kQ - 1) / kQ;
    for (int c = 0; c < nchunks; ++c) {
        const int t0 = c * kQ;
        // S^T (hi and lo) for this chunk's C S product; the previous chunk's MMAs that read it are complete
#pragma unroll
        for (int p = 0; p < kP; ++p) {
            const uint16_t hi = f32_to_bf16(S[p]);
            const uint32_t o = tc::sw128_offset(kP, p, tid);
            *reinterpret_cast<uint16_t*>(sm + kOffSt + o) = hi;
            *reinterpret_cast<uint16_t*>(sm + kOffStLo + o) = f32_to_bf16(S[p] - bf16_to_f32(hi));
        }

        if (tid == 0) {
            mbar_arrive_expect_tx(tma_bar, kTileBytes);
            const int bg = b * a.G + g;
            tma_load_3d(sm + kOffC, &map_c, 0, t0, bg, tma_bar);
            tma_load_3d(sm + kOffC + kQ * 128, &map_c, 64, t0, bg, tma_bar);
            tma_load_3d(sm + kOffB, &map_b, 0, t0, bg, tma_bar);
            tma_load_3d(sm + kOffB + kQ * 128, &map_b, 64, t0, bg, tma_bar);
            tma_load_2d(sm + kOffX, &map_x, t0, static_cast<int>(row0), tma_bar);
            tma_load_2d(sm + kOffX + kP * 128, &map_x, t0 + 64, static_cast<int>(row0), tma_bar);
        }
        tma_pending = true;

        // step sizes and the cumulative decay of the chunk (steps past L: dt = 0, so a = 1 and w = 0)
        const int t = t0 + tid;
        float dtv = 0.0f;
        if (t < L) {
            const float sr = bf16_to_f32(reinterpret_cast<const uint16_t*>(a.dt)[(static_cast<size_t>(b) * a.H + h) * L + t]) + bias;
            dtv = a.softplus ? softplus(sr) : sr;
        }
        float inc = dtv * A2;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += u;
        }
        if (lane == 31) wsum[warp] = inc;
        __syncthreads();
        float s2 = inc;
        for (int w2 = 0; w2 < warp; ++w2) s2 += wsum[w2];
        float w = dtv;
        if (a.zoh && A != 0.0f) w = expm1f(dtv * A) / A;
        s2s[tid] = s2;
        wsv[tid] = w;
        __syncthreads();
        const float s2_end = s2s[kQ - 1];
        vsv[tid] = ex2(s2_end - s2) * w;

        // wait for C, B and X of this chunk
        if (!wait_all(tma_bar, tma_phase)) {
            ok = false;
            break;
        }
        tma_phase ^= 1u;
        tma_pending = false;

        // G = C B^T and C S on the tensor cores
        tc::fence_async_smem();   // S^T written by every thread
        tc::fence_before();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t ko = (ks >> 2) * (kQ * 128) + (ks & 3) * 32;
                tc::mma_bf16(tmem + kColG, tc::desc_k_sw128(sC + ko), tc::desc_k_sw128(sB + ko), tc::idesc_bf16(128, 128),
                             ks > 0);
            }
#pragma unroll
            for (int ks = 0; ks < 16; ++ks) {
                const int k = ks & 7;
                const uint32_t ka = (k >> 2) * (kQ * 128) + (k & 3) * 32;
                const uint32_t kb = (k >> 2) * (kP * 128) + (k & 3) * 32;
                tc::mma_bf16(tmem + kColY1, tc::desc_k_sw128(sC + ka), tc::desc_k_sw128((ks < 8 ? sSt : sStLo) + kb),
                             tc::idesc_bf16(128, kP), ks > 0);
            }
            tc::mma_commit(mma_bar);
        }
        mma_pending = true;

        // meanwhile: row n = tid of the scaled B^T, (exp2(s_end - s_j) w_j B[j, n])_j, hi and lo
#pragma unroll 1
        for (int j0 = 0; j0 < kQ; j0 += 8) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = j0 + 2 * e;
                const float v0 = vsv[j] * ld_bf16_shared(sm + kOffB + tc::sw128_offset(kQ, j, tid));
                const float v1 = vsv[j + 1] * ld_bf16_shared(sm + kOffB + tc::sw128_offset(kQ, j + 1, tid));
                split_pair(v0, v1, hi[e], lo[e]);
            }
            const uint32_t o = tc::sw128_offset(kN, tid, j0);
            st_shared_v4(sm + kOffBt + o, hi[0], hi[1], hi[2], hi[3]);
            st_shared_v4(sm + kOffBtLo + o, lo[0], lo[1], lo[2], lo[3]);
        }

        if (!wait_all(mma_bar, mma_phase)) {
            ok = false;
            break;
        }
        mma_phase ^= 1u;
        mma_pending = false;
        tc::fence_after();

        // row i = tid of M from row i of G (hi into M, lo into the B tile, which G no longer needs)
#pragma unroll 1
        for (int cb = 0; cb < kQ / 32; ++cb) {
            float gv[32];
            tc::tmem_ld32(tmem + tlane + kColG + cb * 32, gv);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = cb * 32 + q * 8 + 2 * e;
                    const float v0 = j <= tid ? gv[q * 8 + 2 * e] * ex2(s2 - s2s[j]) * wsv[j] : 0.0f;
                    const float v1 = j + 1 <= tid ? gv[q * 8 + 2 * e + 1] * ex2(s2 - s2s[j + 1]) * wsv[j + 1] : 0.0f;
                    split_pair(v0, v1, hi[e], lo[e]);
                }
                const uint32_t o = tc::sw128_offset(kQ, tid, cb * 32 + q * 8);
                st_shared_v4(sm + kOffM + o, hi[0], hi[1], hi[2], hi[3]);
                st_shared_v4(sm + kOffMlo + o, lo[0], lo[1], lo[2], lo[3]);
            }
        }
        tc::fence_async_smem();   // M and the scaled B^T
        tc::fence_before();
        __syncthreads();

        // M X and the state increment (scaled B^T) X on the tensor cores
        if (tid == 0) {
            tc::fence_after();
#pragma unroll
            for (int ks = 0; ks < 16; ++ks) {
                const int k = ks & 7;
                const uint32_t ka = (k >> 2) * (kQ * 128) + (k & 3) * 32;
                const uint32_t kb = (k >> 2) * (kP * 128) + (k & 3) * 32;
                tc::mma_bf16(tmem + kColY2, tc::desc_k_sw128((ks < 8 ? sM : sMlo) + ka), tc::desc_k_sw128(sX + kb),
                             tc::idesc_bf16(128, kP), ks > 0);
            }
#pragma unroll
            for (int ks = 0; ks < 16; ++ks) {
                const int k = ks & 7;
                const uint32_t ka = (k >> 2) * (kN * 128) + (k & 3) * 32;
                const uint32_t kb = (k >> 2) * (kP * 128) + (k & 3) * 32;
                tc::mma_bf16(tmem + kColSc, tc::desc_k_sw128((ks < 8 ? sBt : sBtLo) + ka), tc::desc_k_sw128(sX + kb),
                             tc::idesc_bf16(128, kP), ks > 0);
            }
            tc::mma_commit(mma_bar);
        }
        mma_pending = true;
        if (!wait_all(mma_bar, mma_phase)) {
            ok = false;
            break;
        }
        mma_phase ^= 1u;
        mma_pending = false;
        tc::fence_after();

        // outputs of row i = tid (step t)
        const float ei = ex2(s2);
#pragma unroll 1
        for (int pc = 0; pc < kP / 32; ++pc) {
            float y1[32], y2[32];
            tc::tmem_ld32(tmem + tlane + kColY1 + pc * 32, y1);
            tc::tmem_ld32(tmem + tlane + kColY2 + pc * 32, y2);
            if (t < L) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int p = pc * 32 + e;
                    const size_t idx = (row0 + p) * L + t;
                    const float xv = ld_bf16_shared(sm + kOffX + tc::sw128_offset(kP, p, tid));
                    float yv = fmaf(ei, y1[e], y2[e]) + dsk * xv;
                    if (a.z) yv *= silu(bf16_to_f32(reinterpret_cast<const uint16_t*>(a.z)[idx]));
                    reinterpret_cast<uint16_t*>(a.y)[idx] = f32_to_bf16(yv);
                }
            }
        }
        // the state: S <- exp2(s_end) S + increment (row n = tid)
        const float eend = ex2(s2_end);
#pragma unroll
        for (int pc = 0; pc < kP / 32; ++pc) {
            float sc[32];
            tc::tmem_ld32(tmem + tlane + kColSc + pc * 32, sc);
#pragma unroll
            for (int e = 0; e < 32; ++e) S[pc * 32 + e] = fmaf(eend, S[pc * 32 + e], sc[e]);
        }
        tc::fence_before();
        __syncthreads();   // every TMEM and shared read of this chunk is done before the next chunk's copies
    }

    if (ok) {
        if (a.h_out) {
#pragma unroll
            for (int p = 0; p < kP; ++p) a.h_out[(row0 + p) * kN + tid] = S[p];
        }
    } else {
        // a wait gave up: record it, let this block's copies and MMAs still in flight finish (bounded)
        if (tid == 0) {
            atomicOr(&g_ssd_wait_error, 1u);
            if (tma_pending) mbar_wait_bounded(tma_bar, tma_phase);
            if (mma_pending) mbar_wait_bounded(mma_bar, mma_phase);
        }
        tc::fence_before();
        __syncthreads();
    }
    if (warp == 0) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

bool ssd_tc_supported(int N, int P) { return N == kN && P == kP; }

cudaError_t launch_ssd_chunked(const SsdArgs& a, cudaStream_t stream) {
    CUtensorMap mc, mb, mx;
    const uint64_t bc_dims[3] = {static_cast<uint64_t>(kN), static_cast<uint64_t>(a.L),
                                 static_cast<uint64_t>(a.Bsz) * a.G};
    const uint64_t bc_strides[2] = {static_cast<uint64_t>(kN) * 2, static_cast<uint64_t>(a.L) * kN * 2};
    const uint32_t bc_box[3] = {64, kQ, 1};
    const uint64_t x_dims[2] = {static_cast<uint64_t>(a.L), static_cast<uint64_t>(a.Bsz) * a.H * kP};
    const uint64_t x_strides[1] = {static_cast<uint64_t>(a.L) * 2};
    const uint32_t x_box[2] = {64, kP};
    if (!encode_bf16_map_sw128(&mc, a.Cm, 3, bc_dims, bc_strides, bc_box) ||
        !encode_bf16_map_sw128(&mb, a.Bm, 3, bc_dims, bc_strides, bc_box) ||
        !encode_bf16_map_sw128(&mx, a.x, 2, x_dims, x_strides, x_box))
        return cudaErrorInvalidValue;
    cudaError_t e = set_dynamic_smem_once(ssd_chunk_kernel, kSmemBytes);
    if (e != cudaSuccess) return e;
    ssd_chunk_kernel<<<a.Bsz * a.H, kThreads, kSmemBytes, stream>>>(a, mc, mb, mx);
    return cudaGetLastError();
}

cudaError_t take_ssd_wait_error(unsigned* flags) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_ssd_wait_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_ssd_wait_error, &zero, sizeof(unsigned));
}

}  // namespace ssm
