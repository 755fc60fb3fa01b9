// The group quantization rule on the device, shared by every quantizer:
// the E4M3 conversions as the PTX cvt instructions they are, the group
// amax and scale, and the correctly rounded division by the group's scale.
//
// Group rule (quantization table of "NVIDIA强化学习加速实操：10分钟提升2倍训练效率",
// section "为什么FP8适配线性层？": E4M3 codes, FP32 scale per group):
//   amax = max |v|, s = amax / 448 (IEEE division, s = 1 if amax == 0),
//   q = cvt.rn.satfinite.e4m3(fl32(v / s)).
#pragma once

#include <cstdint>

namespace {

// ---------------------------------------------------------------------------
// Conversions, written as the PTX cvt instructions they are.
// ---------------------------------------------------------------------------

// Four E4M3 codes (lowest byte first) -> four exact floats.
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t four, float &a, float &b, float &c,
                                              float &d) {
    asm("{\n\t.reg .b16 lo, hi, h0, h1, h2, h3;\n\t.reg .b32 p, q;\n\t"
        "mov.b32 {lo, hi}, %4;\n\t"
        "cvt.rn.f16x2.e4m3x2 p, lo;\n\t"
        "cvt.rn.f16x2.e4m3x2 q, hi;\n\t"
        "mov.b32 {h0, h1}, p;\n\t"
        "mov.b32 {h2, h3}, q;\n\t"
        "cvt.f32.f16 %0, h0;\n\t"
        "cvt.f32.f16 %1, h1;\n\t"
        "cvt.f32.f16 %2, h2;\n\t"
        "cvt.f32.f16 %3, h3;\n\t}"
        : "=f"(a), "=f"(b), "=f"(c), "=f"(d)
        : "r"(four));
}

// Four floats -> four E4M3 codes (a in the lowest byte): round to nearest
// even, saturating at +-448.
__device__ __forceinline__ uint32_t f32x4_to_e4m3x4(float a, float b, float c, float d) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(a), "f"(b), "f"(c), "f"(d));
    return r;
}

// max(a, |b|, |c|) in one three-input max.
__device__ __forceinline__ float max_abs2(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(fabsf(b)), "f"(fabsf(c)));
    return r;
}

__device__ __forceinline__ float group_scale(float amax) {
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

// ---------------------------------------------------------------------------
// Correctly rounded binary32 division by a group's scale.
//
// Every element of a group is divided by the same s, so the group computes
// y = RN(1/s) once and each quotient costs one multiply and four FMAs
// (Markstein's method; P. Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990):
//   q0 = RN(x*y)                 within 2 ulp of x/s
//   q1 = RN(q0 + RN(x - q0*s)*y) faithful
//   r  = x - q1*s                exact (FMA)
//   q  = RN(q1 + r*y)            = RN(x/s), by Markstein's theorem
// The theorem needs s, 1/s and the residual free of underflow.  s >= 2^-90
// (amax >= 448 * 2^-90) keeps them so for every quotient >= 2^-11; smaller
// quotients can differ from RN(x/s) only far below 2^-10, the smallest E4M3
// rounding boundary, so their codes are the same.  Groups with s < 2^-90
// divide with __fdiv_rn.
//
// The steps run on the negated operands nx = -x and ny = -y:
//   q0 = RN(nx*ny), r' = q0*s + nx = -r (exact), q1 = RN(q0 + r'*ny), ...
// which are the same values with the same roundings, but an exactly zero
// residual now enters the sum as r'*ny with the sign that keeps q's sign of
// zero (x = -0 gives q = -0), so no per-element sign fix-up is needed.
// Callers produce -x directly (a negated scale in a product, or the sign bit
// flipped while widening BF16).
// ---------------------------------------------------------------------------
struct Divisor {
    float s, ny;
    bool fast;
};

__device__ __forceinline__ Divisor make_divisor(float s) {
    Divisor d;
    d.s = s;
    d.fast = s >= 0x1p-90f;
    d.ny = d.fast ? -__frcp_rn(s) : 0.0f;
    return d;
}

// RN(x / s) from nx = -x.
__device__ __forceinline__ float qdiv_neg(float nx, const Divisor &d) {
    if (!d.fast) return __fdiv_rn(-nx, d.s);
    float q = __fmul_rn(nx, d.ny);
    float r = __fmaf_rn(q, d.s, nx);
    q = __fmaf_rn(r, d.ny, q);
    r = __fmaf_rn(q, d.s, nx);
    q = __fmaf_rn(r, d.ny, q);
    return q;
}

// Two quotients with packed f32x2 arithmetic (same steps as qdiv_neg), for a
// divisor known to take the fast path.
__device__ __forceinline__ float2 qdiv2_neg_fast(float2 nx, const Divisor &d) {
    const float2 ny = make_float2(d.ny, d.ny), s = make_float2(d.s, d.s);
    float2 q = __fmul2_rn(nx, ny);
    float2 r = __ffma2_rn(q, s, nx);
    q = __ffma2_rn(r, ny, q);
    r = __ffma2_rn(q, s, nx);
    return __ffma2_rn(r, ny, q);
}

// Four negated values -> four codes of x / s.
__device__ __forceinline__ uint32_t encode4_fast(const float *nf, const Divisor &d) {
    const float2 a = qdiv2_neg_fast(make_float2(nf[0], nf[1]), d);
    const float2 b = qdiv2_neg_fast(make_float2(nf[2], nf[3]), d);
    return f32x4_to_e4m3x4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ uint32_t encode4(const float *nf, const Divisor &d) {
    if (d.fast) return encode4_fast(nf, d);
    return f32x4_to_e4m3x4(qdiv_neg(nf[0], d), qdiv_neg(nf[1], d), qdiv_neg(nf[2], d),
                           qdiv_neg(nf[3], d));
}

}  // namespace
