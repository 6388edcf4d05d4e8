// Single-token decode step, streamed: a persistent kernel that moves the fp32 state cache (B, D, N)
// through shared memory in tiles of 64 (b, d) rows with 1-D bulk copies (the TMA engine) and a ring of
// mbarrier-tracked stages, so that every SM keeps several tiles of loads in flight while it computes
// and stores the previous one.  The step is the scan body with L = 1 (datadaily.news "State space
// models vs Transformer: a practical guide", section on how state space models work: h = Abar h +
// Bbar x_t, y_t = C h + D x_t; cache (batch, d_inner, d_state) per lshu.cn/news/79586 section 6.5).
//
// A tile holds 64 consecutive channels of one batch row: their states and rows of A (N fp32 each),
// their u, delta, z, D skip and dt bias, and the batch row's B and C.  One producer warp issues the
// copies of each tile once the four consumer warps have released its stage (an "empty" mbarrier per
// stage, one arrival per warp); consumers wait on the stage's "full" mbarrier (the copies' byte
// count), so no warp waits on another except through the ring.  A row belongs to 2 consumer threads
// (N / 8 for N > 16), each with 8 consecutive states (4 for N = 8): the per-row scalars (softplus,
// gate, conv) are computed by few threads, and a warp still reads and writes whole rows of the state.
// The new state leaves with 16-byte streaming stores straight from registers; y leaves from the first
// thread of each row.
//
// Requirements (the host checks them before choosing this kernel): N in {8, 16, 32, 64}, D % 8 == 0
// (every tile's row count is a multiple of 8, so every copy is a multiple of 16 bytes) and 16-byte
// aligned state, A, u, delta, z, B, C, D skip and dt bias.
//
// Each wait on a stage is bounded (about one second).  On a timeout the warp records it in a flag that
// ssm_device_error reads and stops; before the block leaves, one thread waits (bounded) for the copies
// it issued but did not consume.
#include <algorithm>
#include <type_traits>

#include "bulk_copy.cuh"
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

namespace {

constexpr int kBulkThreads = 128;

__device__ unsigned int g_bulk_wait_error = 0;

constexpr int round16(int x) { return (x + 15) & ~15; }

template <typename T, int N, bool kConv>
struct BulkLayout {
    // rows of (b, d) per tile and tiles in flight per block: for N <= 16 two 128-row tiles beat four 64-row
    // ones (fewer, longer copies per barrier round trip); wider states keep 64-row tiles so that several
    // blocks still fit on an SM
    static constexpr int kTileRows = N <= 16 ? 128 : 64;
    static constexpr int kE = T::kBytes;
    static constexpr int kState = kTileRows * N * 4;
    static constexpr int kScal = round16(kTileRows * kE);
    static constexpr int kBC = round16(N * kE);
    static constexpr int kOffState = 0;
    static constexpr int kOffA = kOffState + kState;
    static constexpr int kOffU = kOffA + kState;
    static constexpr int kOffDt = kOffU + kScal;
    static constexpr int kOffZ = kOffDt + kScal;
    static constexpr int kOffB = kOffZ + kScal;
    static constexpr int kOffC = kOffB + kBC;
    static constexpr int kOffD = kOffC + kBC;
    static constexpr int kOffBias = kOffD + kTileRows * 4;
    // conv front end (kConv): the rows' conv states (W - 1 <= 3 inputs each), taps (W <= 4) and biases
    static constexpr int kOffCS = round16(kOffBias + kTileRows * 4);
    static constexpr int kOffCW = kOffCS + (kConv ? round16(kTileRows * 3 * kE) : 0);
    static constexpr int kOffCB = kOffCW + (kConv ? kTileRows * 4 * 4 : 0);
    static constexpr int kBytes = round16(kOffCB + (kConv ? kTileRows * 4 : 0));
    static constexpr int kStages = N <= 16 ? 2 : (N <= 32 ? 4 : 3);
    static constexpr int kSmem = 128 + kStages * kBytes;  // barriers and counters first
};

struct DecodeArgs {
    float* state;
    const void* u;
    const void* delta;
    const float* A;
    const void* Bm;
    const void* Cm;
    const float* Dskip;
    const float* delta_bias;
    const void* z;
    void* y;
    const float* conv_w;  // (D, W) or NULL
    const float* conv_b;  // (D) or NULL
    void* conv_state;     // (B, D, W - 1), read and written; NULL when W == 1
    int W;
    const int* state_indices;  // (B) slot of each batch row in state / conv_state, or NULL (slot = b)
    int Bsz, D, softplus;
    int withhold;              // test only: block 0 never copies its first tile (its waits run out)
};

template <typename T>
__device__ __forceinline__ float smem_scalar(const unsigned char* base, int i) {
    if constexpr (T::kBytes == 4) {
        return reinterpret_cast<const float*>(base)[i];
    } else {
        return bf16_to_f32(reinterpret_cast<const uint16_t*>(base)[i]);
    }
}

template <typename T>
__device__ __forceinline__ void smem_vec4(const unsigned char* base, int i, float (&v)[4]) {
    if constexpr (T::kBytes == 4) {
        const float4 w = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + i);
        v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
    } else {
        const uint2 w = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(base) + i);
        v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    }
}

template <typename T, int N, bool kZOH, bool kConv>
__global__ void __launch_bounds__(kBulkThreads + 32, 4) state_update_bulk_kernel(const DecodeArgs a) {
    using L = BulkLayout<T, N, kConv>;
    constexpr int S = L::kStages;
    constexpr int kTileRows = L::kTileRows;
    constexpr int E = L::kE;
    constexpr int TPR = N <= 16 ? 2 : N / 8;   // threads per row
    constexpr int SL = N / TPR;                 // states per thread: 4 (N = 8) or 8
    constexpr int RPP = kBulkThreads / TPR;     // rows per pass
    constexpr int kWarps = kBulkThreads / 32;   // consumer warps
    extern __shared__ __align__(128) unsigned char bulk_smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(bulk_smem);   // copies of a stage landed
    uint64_t* empty = full + S;                                // every consumer warp is done with a stage
    int* counts = reinterpret_cast<int*>(empty + S);           // [0] tiles issued, [1 + w] tiles consumed by warp w
    unsigned char* stages = bulk_smem + 128;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int tiles_per_b = (a.D + kTileRows - 1) / kTileRows;
    const int total = a.Bsz * tiles_per_b;
    const int G = gridDim.x;
    const int nlocal = (int)blockIdx.x < total ? (total - 1 - (int)blockIdx.x) / G + 1 : 0;

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        mbar_fence_init();
    }
    pdl_wait();     // the previous kernel of the stream is done: its outputs may be this call's inputs
    pdl_release();
    __syncthreads();

    if (warp == kWarps) {
        // producer warp: one lane streams the block's tiles into the stage ring
        if (lane == 0) {
            int j = 0;
            for (; j < nlocal; ++j) {
                const int s = j % S;
                if (j >= S && !mbar_wait_bounded(&empty[s], (unsigned)((j / S - 1) & 1))) {
                    atomicOr(&g_bulk_wait_error, 1u);
                    break;
                }
                if (a.withhold && blockIdx.x == 0 && j == 0) continue;   // no copy, no arrival: a wait runs out
                const int t = (int)blockIdx.x + j * G;
                const int b = t / tiles_per_b;
                const int d0 = (t - b * tiles_per_b) * kTileRows;
                const int rows = min(kTileRows, a.D - d0);
                const size_t r0 = (size_t)b * a.D + d0;
                uint64_t* bar = &full[s];
                unsigned char* st = stages + s * L::kBytes;
                const int slot = a.state_indices != nullptr ? __ldg(a.state_indices + b) : b;
                if (slot < 0) {  // a padding row: nothing to copy, the stage is complete at once
                    mbar_arrive(bar);
                    continue;
                }
                const size_t s0 = (size_t)slot * a.D + d0;  // the tile's first row in the state cache
                const unsigned sb = (unsigned)(rows * N * 4), eb = (unsigned)(rows * E), pb = (unsigned)(rows * 4);
                unsigned bytes = 2 * sb + 2 * eb + (a.z ? eb : 0u) + 2u * N * E + (a.Dskip ? pb : 0u) +
                                 (a.delta_bias ? pb : 0u);
                const unsigned csb = (unsigned)(rows * (a.W - 1) * E), cwb = (unsigned)(rows * a.W * 4);
                if (kConv) bytes += (a.W > 1 ? csb : 0u) + cwb + (a.conv_b ? pb : 0u);
                mbar_arrive_expect_tx(bar, bytes);
                if (kConv) {
                    if (a.W > 1)
                        bulk_g2s(st + L::kOffCS, static_cast<const unsigned char*>(a.conv_state) + s0 * (a.W - 1) * E,
                                 csb, bar);
                    bulk_g2s(st + L::kOffCW, a.conv_w + (size_t)d0 * a.W, cwb, bar);
                    if (a.conv_b) bulk_g2s(st + L::kOffCB, a.conv_b + d0, pb, bar);
                }
                bulk_g2s(st + L::kOffState, a.state + s0 * N, sb, bar);
                bulk_g2s(st + L::kOffA, a.A + (size_t)d0 * N, sb, bar);
                bulk_g2s(st + L::kOffU, static_cast<const unsigned char*>(a.u) + r0 * E, eb, bar);
                bulk_g2s(st + L::kOffDt, static_cast<const unsigned char*>(a.delta) + r0 * E, eb, bar);
                if (a.z) bulk_g2s(st + L::kOffZ, static_cast<const unsigned char*>(a.z) + r0 * E, eb, bar);
                bulk_g2s(st + L::kOffB, static_cast<const unsigned char*>(a.Bm) + (size_t)b * N * E, N * E, bar);
                bulk_g2s(st + L::kOffC, static_cast<const unsigned char*>(a.Cm) + (size_t)b * N * E, N * E, bar);
                if (a.Dskip) bulk_g2s(st + L::kOffD, a.Dskip + d0, pb, bar);
                if (a.delta_bias) bulk_g2s(st + L::kOffBias, a.delta_bias + d0, pb, bar);
            }
            counts[0] = j;
        }
    } else {
        const int q = tid % TPR;
        int j = 0;
        for (; j < nlocal; ++j) {
            const int s = j % S;
            if (!mbar_wait_bounded(&full[s], (unsigned)((j / S) & 1))) {
                if (lane == 0) atomicOr(&g_bulk_wait_error, 1u);
                break;
            }
            const int t = (int)blockIdx.x + j * G;
            const int b = t / tiles_per_b;
            const int d0 = (t - b * tiles_per_b) * kTileRows;
            const int rows = min(kTileRows, a.D - d0);
            const size_t r0 = (size_t)b * a.D + d0;
            const int slot = a.state_indices != nullptr ? __ldg(a.state_indices + b) : b;
            if (slot < 0) {  // a padding row: y = 0, no slot touched
                for (int r = tid / TPR; r < rows; r += RPP)
                    if (q == 0) store1<T>(a.y, r0 + r, 0.0f);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                continue;
            }
            const size_t s0 = (size_t)slot * a.D + d0;
            const unsigned char* st = stages + s * L::kBytes;
            const float* hs = reinterpret_cast<const float*>(st + L::kOffState);
            const float* As = reinterpret_cast<const float*>(st + L::kOffA);
            const float* Ds = reinterpret_cast<const float*>(st + L::kOffD);
            const float* bs = reinterpret_cast<const float*>(st + L::kOffBias);
            // this thread's states are SL * q .. SL * q + SL - 1 (whole 16-byte chunks of a row)
            float Bv[SL], Cv[SL];
#pragma unroll
            for (int c = 0; c < SL / 4; ++c) {
                float t4[4];
                smem_vec4<T>(st + L::kOffB, SL * q + 4 * c, t4);
#pragma unroll
                for (int i = 0; i < 4; ++i) Bv[4 * c + i] = t4[i];
                smem_vec4<T>(st + L::kOffC, SL * q + 4 * c, t4);
#pragma unroll
                for (int i = 0; i < 4; ++i) Cv[4 * c + i] = t4[i];
            }
            // bf16 I/O: a warp whose rows in this tile all have |A| >= kZohFastMinA takes the fast zero-order-
            // hold form (its error is far inside the bf16 bound there); fp32 I/O always the exact form.  One
            // vote per tile and warp, and the row loop instantiated once per form: a per-row choice inside
            // the unrolled loop measured 5 % slower than either form alone.
            bool exact = T::kBytes != 2;
            if (kZOH && !exact) {
                bool small_a = false;
#pragma unroll
                for (int p = 0; p < kTileRows / RPP; ++p) {
                    const int r = p * RPP + tid / TPR;  // rows past the tile's end hold stale values: harmless
#pragma unroll
                    for (int c = 0; c < SL / 4; ++c) {
                        const float4 av = *reinterpret_cast<const float4*>(As + r * N + SL * q + 4 * c);
                        small_a |= !(fabsf(av.x) >= kZohFastMinA) || !(fabsf(av.y) >= kZohFastMinA) ||
                                   !(fabsf(av.z) >= kZohFastMinA) || !(fabsf(av.w) >= kZohFastMinA);
                    }
                }
                exact = __any_sync(0xffffffffu, small_a);
            }
            auto rows_pass = [&](auto exact_form) {
                constexpr bool kExact = decltype(exact_form)::value;
    #pragma unroll
                for (int p = 0; p < kTileRows / RPP; ++p) {
                    // every lane takes part in the shuffles; rows past the tile's end compute on stale values
                    // and store nothing
                    const int r = p * RPP + tid / TPR;
                    float h[SL], A4[SL];
    #pragma unroll
                    for (int c = 0; c < SL / 4; ++c) {
                        const float4 hv = *reinterpret_cast<const float4*>(hs + r * N + SL * q + 4 * c);
                        const float4 av = *reinterpret_cast<const float4*>(As + r * N + SL * q + 4 * c);
                        h[4 * c] = hv.x; h[4 * c + 1] = hv.y; h[4 * c + 2] = hv.z; h[4 * c + 3] = hv.w;
                        A4[4 * c] = av.x; A4[4 * c + 1] = av.y; A4[4 * c + 2] = av.z; A4[4 * c + 3] = av.w;
                    }
                    float uv = smem_scalar<T>(st + L::kOffU, r);
                    if constexpr (kConv) {
                        // v = SiLU(conv_b + sum_k w_k x_{t-W+1+k}); x before t is the row's conv state
                        const int W1 = a.W - 1;
                        const float* cw = reinterpret_cast<const float*>(st + L::kOffCW) + r * a.W;
                        float c = a.conv_b ? reinterpret_cast<const float*>(st + L::kOffCB)[r] : 0.0f;
    #pragma unroll
                        for (int k = 0; k < 3; ++k)
                            if (k < W1) c = fmaf(cw[k], smem_scalar<T>(st + L::kOffCS, r * W1 + k), c);
                        c = fmaf(cw[W1], uv, c);
                        if (q == 0 && r < rows) {
                            // the new conv state: the last W - 1 inputs, oldest first (raw values, no rounding)
                            using Sx = typename T::storage;
                            const Sx* cs = reinterpret_cast<const Sx*>(st + L::kOffCS) + r * W1;
                            Sx* out = static_cast<Sx*>(a.conv_state) + (s0 + r) * W1;
    #pragma unroll
                            for (int k = 0; k < 3; ++k)
                                if (k < W1) out[k] = k + 1 < W1 ? cs[k + 1] : reinterpret_cast<const Sx*>(st + L::kOffU)[r];
                        }
                        if constexpr (T::kBytes == 2) uv = silu_fast(c);
                        else uv = silu(c);
                    }
                    const float sr = smem_scalar<T>(st + L::kOffDt, r) + (a.delta_bias ? bs[r] : 0.0f);
                    const float zr = a.z ? smem_scalar<T>(st + L::kOffZ, r) : 0.0f;
                    const float dsk = a.Dskip ? Ds[r] : 0.0f;
                    float dt, gate;
                    if constexpr (T::kBytes == 2) {  // bf16 I/O: the MUFU forms
                        dt = a.softplus ? softplus_fast(sr) : sr;
                        gate = a.z ? silu_fast(zr) : 1.0f;
                    } else {
                        dt = a.softplus ? softplus(sr) : sr;
                        gate = a.z ? silu(zr) : 1.0f;
                    }
                    const float dtu = dt * uv;
                    float yp = 0.0f;
    #pragma unroll
                    for (int i = 0; i < SL; ++i) {
                        const float y = dt * (A4[i] * kLog2e);
                        if (kZOH && kExact) {
                            // exact form, branch-free: E (and Abar) from the series where |dt a| < 2^-4 (dt at
                            // a = 0)
                            float ab;
                            const float E = zoh_exact(dt, y, A4[i] != 0.0f ? rcp(A4[i]) : 0.0f, ab);
                            h[i] = fmaf(ab, h[i], E * (uv * Bv[i]));
                        } else if (kZOH) {
                            // fast form h' = Abar (h - ng) + ng, ng = -(v / a) B (every |a| >= 1/4 in the warp)
                            const float ng = (uv * -rcp(A4[i])) * Bv[i];
                            h[i] = fmaf(ex2(y), h[i] - ng, ng);
                        } else {
                            h[i] = fmaf(abar_exact(y), h[i], dtu * Bv[i]);
                        }
                        yp = fmaf(Cv[i], h[i], yp);
                    }
    #pragma unroll
                    for (int m = 1; m < TPR; m <<= 1) yp += __shfl_xor_sync(0xffffffffu, yp, m);
                    if (r < rows) {
    #pragma unroll
                        for (int c = 0; c < SL / 4; ++c)
                            __stcs(reinterpret_cast<float4*>(a.state + (s0 + r) * N + SL * q + 4 * c),
                                   make_float4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]));
                        if (q == 0) store1<T>(a.y, r0 + r, fmaf(dsk, uv, yp) * gate);
                    }
                }
            };
            if (exact) rows_pass(std::true_type{});
            else rows_pass(std::false_type{});
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (lane == 0) counts[1 + warp] = j;
    }

    __syncthreads();
    if (tid == 0) {
        // after a timeout, let the copies this block issued but did not consume land before it leaves
        int consumed = nlocal;
        for (int w = 0; w < kWarps; ++w) consumed = min(consumed, counts[1 + w]);
        for (int jj = consumed; jj < counts[0]; ++jj) mbar_wait_bounded(&full[jj % S], (unsigned)((jj / S) & 1));
    }
}

template <typename T, int N, bool kZOH, bool kConv>
cudaError_t launch_bulk(const DecodeArgs& a, cudaStream_t stream) {
    using L = BulkLayout<T, N, kConv>;
    auto kfn = state_update_bulk_kernel<T, N, kZOH, kConv>;
    cudaError_t e = set_dynamic_smem_once(kfn, L::kSmem);
    if (e != cudaSuccess) return e;
    int slots = 0;  // resident blocks on the whole device, asked once per kernel and device
    if ((e = resident_blocks(reinterpret_cast<const void*>(kfn), kBulkThreads + 32, L::kSmem, &slots)) != cudaSuccess)
        return e;
    const long long tiles = (long long)a.Bsz * ((a.D + L::kTileRows - 1) / L::kTileRows);
    const int grid = (int)std::min<long long>(tiles, (long long)std::max(slots, 1));
    e = launch_pdl(kfn, dim3(grid), dim3(kBulkThreads + 32), L::kSmem, stream, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename T, int N>
cudaError_t launch_bulk_n(const DecodeArgs& a, int zoh, cudaStream_t s) {
    if (a.conv_w != nullptr) return zoh ? launch_bulk<T, N, true, true>(a, s) : launch_bulk<T, N, false, true>(a, s);
    return zoh ? launch_bulk<T, N, true, false>(a, s) : launch_bulk<T, N, false, false>(a, s);
}

template <typename T>
cudaError_t launch_bulk_t(const DecodeArgs& a, int N, int zoh, cudaStream_t s) {
    switch (N) {
        case 8: return launch_bulk_n<T, 8>(a, zoh, s);
        case 16: return launch_bulk_n<T, 16>(a, zoh, s);
        case 32: return launch_bulk_n<T, 32>(a, zoh, s);
        default: return launch_bulk_n<T, 64>(a, zoh, s);
    }
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

bool state_update_bulk_eligible(const DecodeStep& s) {
    if (s.N != 8 && s.N != 16 && s.N != 32 && s.N != 64) return false;
    if (s.D % 8 != 0) return false;
    const bool conv_ok = !s.conv_w || (al16(s.conv_w) && (!s.conv_b || al16(s.conv_b)) &&
                                       (s.conv_width == 1 || al16(s.conv_state)));
    return al16(s.state) && al16(s.x) && al16(s.delta) && al16(s.A) && al16(s.Bm) && al16(s.Cm) &&
           (!s.Dskip || al16(s.Dskip)) && (!s.delta_bias || al16(s.delta_bias)) && (!s.z || al16(s.z)) && conv_ok;
}

cudaError_t launch_state_update_bulk(const DecodeStep& s, cudaStream_t stream) {
    const DecodeArgs a{s.state, s.x, s.delta, s.A, s.Bm, s.Cm, s.Dskip, s.delta_bias, s.z, s.y,
                       s.conv_w, s.conv_w ? s.conv_b : nullptr, s.conv_w ? s.conv_state : nullptr,
                       s.conv_w ? s.conv_width : 1, s.state_indices, s.Bsz, s.D, s.softplus,
                       withhold_first_copy() ? 1 : 0};
    if (s.dtype == 1) return launch_bulk_t<BF16>(a, s.N, s.zoh, stream);
    return launch_bulk_t<F32>(a, s.N, s.zoh, stream);
}

cudaError_t take_bulk_wait_error(unsigned* flags) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_bulk_wait_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_bulk_wait_error, &zero, sizeof(unsigned));
}

}  // namespace ssm
