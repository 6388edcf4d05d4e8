// Device-side helpers shared by the scan, conv and decode kernels: MUFU wrappers, the step-size
// softplus, SiLU, and bf16 / fp32 vector loads and stores.  sm_103a only.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Discretisation of the input term: zero-order hold, zero-order hold with A == 0 entries present in
// the warp (uses the dt * B limit there), or the simplified dt * B.
enum class Disc { kZOH, kZOHSafe, kSimple };

// 2^x on the MUFU unit (ex2.approx.ftz: about 2 ulp, 32 results per clock per SM on B300).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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
