// Device-side helpers shared by the scan, conv and decode kernels: MUFU wrappers, the step-size
// softplus, SiLU, and bf16 / fp32 vector loads and stores.  sm_103a only.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Discretisation of the input term: zero-order hold in the fast form (for blocks whose every state
// has |A| >= kZohFastMinA), zero-order hold in the exact form (any A, including 0), or the
// simplified dt * B.
enum class Disc { kZOH, kZOHExact, kSimple };

// ---------------------------------------------------------------------------------------------
// Zero-order hold input factor E = (exp(x) - 1) / a, x = dt a (dpshk.com/news/3333417 section 2.2,
// lshu.cn/news/79586 section 2.2, diagonal A), so that Bbar = E B.
//
// Formed as (Abar - 1) / a, E loses log2(1/|x|) bits to cancellation: Abar carries an absolute
// error of about 2^-23 near 1, so E's relative error is about 1.2e-7 / |x|.  Below |x| = 2^-4 the
// exact form is used instead: E = dt phi(x), phi(x) = expm1(x) / x = sum_k x^k / (k+1)!, summed
// by Horner to the x^3 term (truncation x^4 / 120 < 1.3e-7 relative at |x| = 2^-4).  Above the
// threshold (Abar - 1) / a is within about 4e-6 relative.  At a = 0 the series gives the limit dt.
// The series and the threshold are written from the Taylor expansion of exp, not from any library.
// ---------------------------------------------------------------------------------------------
constexpr float kZohSeriesX = 0.0625f;              // |x| below which E comes from the series
constexpr float kZohSeriesY = 0.0625f * kLog2e;     // the same threshold for y = x log2(e)
// phi(x) = 1 + x/2 + x^2/6 + x^3/24 written in y = x log2 e: coefficients (ln 2)^k / (k+1)!
constexpr float kPhiY1 = 0.34657359027997264f;      // ln2 / 2
constexpr float kPhiY2 = 0.08007550231970023f;      // ln2^2 / 6
constexpr float kPhiY3 = 0.013876027166205394f;     // ln2^3 / 24
// Blocks (warps) in which every state has |A| at least this may use the fast form
// h' = Abar (h - ng) + ng, ng = -(v / a) B: its absolute error per step is about 2^-22 |v B / a|, so
// over the at most 64 k steps that a state remembers it stays near 2.5e-4 |v B| for |A| >= 1/4, within
// the bf16-path state bound 1e-3 (1 + |h|).  The fp32 path always takes the exact form.
constexpr float kZohFastMinA = 0.25f;

// phi(x) in terms of y = x log2 e (|y| < kZohSeriesY).
__device__ __forceinline__ float zoh_phi_y(float y) {
    float p = fmaf(y, kPhiY3, kPhiY2);
    p = fmaf(p, y, kPhiY1);
    return fmaf(p, y, 1.0f);
}

// E for one state: y = dt a log2 e, ab = 2^y, inva = 1 / a (0 where a == 0).
__device__ __forceinline__ float zoh_factor(float dt, float y, float ab, float inva) {
    const float big = (ab - 1.0f) * inva;
    const float small = dt * zoh_phi_y(y);
    return fabsf(y) < kZohSeriesY ? small : big;
}

// dE/da for the backward pass: (dt Abar - E) / a, which cancels twice as x -> 0 (dt Abar - E is about
// dt x / 2), so below |x| = 1/4 it is dt^2 phi'(x), phi'(x) = sum_k k x^(k-1) / (k+1)!
// = 1/2 + x/3 + x^2/8 + x^3/30 + x^4/144 + x^5/840 (truncation x^6 / 5760 < 1e-7 relative at |x| = 1/4);
// above, the quotient is within about 1e-5 relative.
constexpr float kZohDaSeriesX = 0.25f;
__device__ __forceinline__ float zoh_factor_da(float dt, float x, float ab, float E, float inva) {
    const float big = fmaf(dt, ab, -E) * inva;
    float p = fmaf(x, 1.0f / 840.0f, 1.0f / 144.0f);
    p = fmaf(p, x, 1.0f / 30.0f);
    p = fmaf(p, x, 0.125f);
    p = fmaf(p, x, 1.0f / 3.0f);
    p = fmaf(p, x, 0.5f);
    const float small = dt * dt * p;
    return fabsf(x) < kZohDaSeriesX ? small : big;
}

// 2^x on the MUFU unit (ex2.approx.ftz: about 2 ulp, 32 results per clock per SM on B300).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Abar and E of the exact form together, for the kernels whose states carry fp32 accuracy over long
// sequences (the fp32-output scan, the decode step): where the series holds, Abar = 1 + x phi(x) (x = y ln 2)
// comes within about half an ulp of e^x, where the ~2 ulp of ex2.approx would build up over the thousands
// of steps that such a state remembers; elsewhere 2^y and (2^y - 1) / a.  inva = 1 / a (0 where a == 0).
__device__ __forceinline__ float zoh_exact(float dt, float y, float inva, float& ab) {
    const float phi = zoh_phi_y(y);
    const float e = ex2(y);
    const bool series = fabsf(y) < kZohSeriesY;
    ab = series ? fmaf(y * kLn2, phi, 1.0f) : e;
    return series ? dt * phi : (e - 1.0f) * inva;
}

// Abar alone the same way, for the simplified input scale (Bbar = dt B) on those kernels.
__device__ __forceinline__ float abar_exact(float y) {
    return fabsf(y) < kZohSeriesY ? fmaf(y * kLn2, zoh_phi_y(y), 1.0f) : ex2(y);
}

// 1/x on the MUFU unit (rcp.approx.ftz: about 1 ulp).
__device__ __forceinline__ float rcp(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log1p(e) for e in [0, 1]: e * P(e) with the degree-8 least-squares polynomial made by
// gen_log1p_poly.py (max relative error 1.9e-7 in fp32 Horner form).  The MUFU log is not used
// because its error is absolute, which near 1 destroys the relative accuracy of small log1p.
__device__ __forceinline__ float log1p_unit(float e) {
    float p = 0.005253457929939032f;
    p = fmaf(p, e, -0.02958850748836994f);
    p = fmaf(p, e, 0.07836166769266129f);
    p = fmaf(p, e, -0.13674770295619965f);
    p = fmaf(p, e, 0.19111430644989014f);
    p = fmaf(p, e, -0.24844369292259216f);
    p = fmaf(p, e, 0.33319270610809326f);
    p = fmaf(p, e, -0.49999502301216125f);
    p = fmaf(p, e, 1.0f);
    return p * e;
}

// softplus(s) = log(1 + e^s) = max(s, 0) + log1p(e^-|s|): no overflow, no cancellation.
__device__ __forceinline__ float softplus(float s) {
    float e = ex2(-fabsf(s) * kLog2e);
    return fmaxf(s, 0.0f) + log1p_unit(e);
}

// SiLU(v) = v * sigmoid(v) = v / (1 + e^-v).  For v < -88 the exponential overflows to +inf and
// the reciprocal gives 0, the correctly rounded limit.
__device__ __forceinline__ float silu(float v) {
    return v * rcp(1.0f + ex2(-v * kLog2e));
}

// Variants for bf16 outputs (whose rounding is 2^-9): they move work from the FMA pipe to the
// MUFU, which the scan kernels have to spare.
// tanh on the MUFU (tanh.approx: relative error about 1e-5, 16 results per clock per SM on B300).
__device__ __forceinline__ float tanh_mufu(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// log2 on the MUFU (lg2.approx: absolute error about 2e-7 near 1).
__device__ __forceinline__ float lg2_mufu(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// SiLU(v) = v sigmoid(v) = h + h tanh(h) with h = v / 2.
__device__ __forceinline__ float silu_fast(float v) {
    const float hv = 0.5f * v;
    return fmaf(hv, tanh_mufu(hv), hv);
}
// softplus(s) = max(s, 0) + ln2 * log2(1 + 2^(-|s| log2 e)); absolute error about 2e-7.
__device__ __forceinline__ float softplus_fast(float s) {
    const float e = ex2(-fabsf(s) * kLog2e);
    return fmaf(lg2_mufu(1.0f + e), kLn2, fmaxf(s, 0.0f));
}

// ---------------------------------------------------------------------------------------------
// Packed pairs of fp32 (sm_100+ f32x2 instructions): one issue slot for two lanes of FMA-pipe work.
// ---------------------------------------------------------------------------------------------
using f32x2 = unsigned long long;

__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(f32x2 v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
    f32x2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ f32x2 ex2x2(f32x2 x) {
    float a, b;
    unpack2(x, a, b);
    return pack2(ex2(a), ex2(b));
}

// zoh_factor on a pair of states, given ninv2 = -1/a (0 where a == 0): series and quotient both on
// packed pairs, the choice per state.
__device__ __forceinline__ f32x2 zoh_factor2(f32x2 dt2, f32x2 y2, f32x2 ab2, f32x2 ninv2) {
    f32x2 p = fma2(y2, pack2(kPhiY3, kPhiY3), pack2(kPhiY2, kPhiY2));
    p = fma2(p, y2, pack2(kPhiY1, kPhiY1));
    p = fma2(p, y2, pack2(1.0f, 1.0f));
    const f32x2 small = mul2(p, dt2);
    const f32x2 big = mul2(sub2(pack2(1.0f, 1.0f), ab2), ninv2);
    float y0, y1, s0, s1, b0, b1;
    unpack2(y2, y0, y1);
    unpack2(small, s0, s1);
    unpack2(big, b0, b1);
    return pack2(fabsf(y0) < kZohSeriesY ? s0 : b0, fabsf(y1) < kZohSeriesY ? s1 : b1);
}

// zoh_factor_da on a pair of states (the same series, coefficients and threshold): x2 = dt a, dt22 = dt^2,
// E2 = zoh_factor2(...), inva2 = 1/a (0 where a == 0).
__device__ __forceinline__ f32x2 zoh_factor_da2(f32x2 dt2, f32x2 dt22, f32x2 x2, f32x2 ab2, f32x2 E2, f32x2 inva2) {
    const f32x2 big = mul2(fma2(dt2, ab2, mul2(E2, pack2(-1.0f, -1.0f))), inva2);  // one rounding, as fmaf
    f32x2 p = fma2(x2, pack2(1.0f / 840.0f, 1.0f / 840.0f), pack2(1.0f / 144.0f, 1.0f / 144.0f));
    p = fma2(p, x2, pack2(1.0f / 30.0f, 1.0f / 30.0f));
    p = fma2(p, x2, pack2(0.125f, 0.125f));
    p = fma2(p, x2, pack2(1.0f / 3.0f, 1.0f / 3.0f));
    p = fma2(p, x2, pack2(0.5f, 0.5f));
    const f32x2 small = mul2(dt22, p);
    float x0, x1, s0, s1, b0, b1;
    unpack2(x2, x0, x1);
    unpack2(small, s0, s1);
    unpack2(big, b0, b1);
    return pack2(fabsf(x0) < kZohDaSeriesX ? s0 : b0, fabsf(x1) < kZohDaSeriesX ? s1 : b1);
}

// ---------------------------------------------------------------------------------------------
// bf16 <-> fp32.  bf16 is the top half of an fp32, so widening is a shift; narrowing rounds to
// nearest even with cvt.rn.bf16x2.f32.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    return static_cast<uint16_t>(pack_bf16x2(f, 0.0f) & 0xffffu);
}

// Element type tags.
struct F32 {
    using storage = float;
    static constexpr int kBytes = 4;
};
struct BF16 {
    using storage = uint16_t;
    static constexpr int kBytes = 2;
};

template <typename T>
__device__ __forceinline__ float load1(const void* base, size_t i);
template <>
__device__ __forceinline__ float load1<F32>(const void* base, size_t i) {
    return __ldg(static_cast<const float*>(base) + i);
}
template <>
__device__ __forceinline__ float load1<BF16>(const void* base, size_t i) {
    return bf16_to_f32(__ldg(static_cast<const uint16_t*>(base) + i));
}

template <typename T>
__device__ __forceinline__ void store1(void* base, size_t i, float v);
template <>
__device__ __forceinline__ void store1<F32>(void* base, size_t i, float v) {
    static_cast<float*>(base)[i] = v;
}
template <>
__device__ __forceinline__ void store1<BF16>(void* base, size_t i, float v) {
    static_cast<uint16_t*>(base)[i] = f32_to_bf16(v);
}

// 8 consecutive elements starting at element i, with 16-byte vector loads (caller guarantees
// 16-byte alignment of base + i).  Streaming data: read once, keep it out of L1.
template <typename T>
__device__ __forceinline__ void load8(const void* base, size_t i, float (&v)[8]);
template <>
__device__ __forceinline__ void load8<F32>(const void* base, size_t i, float (&v)[8]) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + i);
    float4 a = __ldcs(p), b = __ldcs(p + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<BF16>(const void* base, size_t i, float (&v)[8]) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + i);
    uint4 w = __ldcs(p);
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x);
    v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z);
    v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
}

template <typename T>
__device__ __forceinline__ void store8(void* base, size_t i, const float (&v)[8]);
template <>
__device__ __forceinline__ void store8<F32>(void* base, size_t i, const float (&v)[8]) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + i);
    __stcs(p, make_float4(v[0], v[1], v[2], v[3]));
    __stcs(p + 1, make_float4(v[4], v[5], v[6], v[7]));
}
template <>
__device__ __forceinline__ void store8<BF16>(void* base, size_t i, const float (&v)[8]) {
    uint4 w;
    w.x = pack_bf16x2(v[0], v[1]);
    w.y = pack_bf16x2(v[2], v[3]);
    w.z = pack_bf16x2(v[4], v[5]);
    w.w = pack_bf16x2(v[6], v[7]);
    __stcs(reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + i), w);
}

}  // namespace ssm
