// SwiGLU with the 1x128 quantization of its output fused: the MLP's down
// projection input is written as FP8 codes and scales straight from the
// gate and up products, with no BF16 activation in between.  The pages fuse
// the quantizer into the operator that produces a linear layer's input
// ("英伟达破解AI训练效率难题" (163.com), section 三; "Jet-RL ..." (gist.science),
// "Quantisierungsschema"); for the down projection that operator is SwiGLU,
// h = silu(gate) * up.
//
// Arithmetic (the binary32 operations of the specification of this operator,
// every step one IEEE operation with round-to-nearest, none contracted, run
// two elements at a time with packed f32x2 instructions; the changes of form
// listed at neg_swiglu_f32x2 give the same bits):
//   e^x  : Cody-Waite reduction x = n ln2 + r with ln 2 split into a 16-bit
//          head and a rounded tail (fused multiply-adds), the Taylor
//          polynomial of e^r to degree 7 in Horner form with coefficients
//          RN(1/k!), and the scaling by 2^(n/2) then 2^(n - n/2) (truncating
//          division), both exact powers of two.
//   silu : g < -80 gives g * 0; otherwise d = 1 + e^max(-g, -104), 1/d from
//          the bit-pattern seed 0x7EF311C7 - bits(d) and three Newton-Raphson
//          steps y += y (1 - d y), silu = g * y.
//   h    : silu(g) * up, then the 1x128 group rule of quant_rule.cuh on the
//          binary32 values of h.
//
// One warp takes one row and two consecutive 128-wide groups of it (lanes
// 0-15 the first, 16-31 the second; 8 elements per lane, one 16-byte load of
// gate and of up); consecutive warps take consecutive rows of the same two
// groups, so that the warps of a CTA write their scales next to each other.
// Each warp loads its next item before computing the current one.  At 4 bytes
// in and 1 + 4/128 out per element the kernel would be bound by HBM; with
// about 40 instructions per element it is bound by instruction issue.
#include <cuda_bf16.h>

#include "jet_common.cuh"
#include "stream_ld.cuh"
#include "quant_rule.cuh"

namespace {

constexpr int kSwThreads = 256;
constexpr int kSwCtasPerSm = 4;
__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

// e^x for two arguments in [-87, 80], packed f32x2 arithmetic.  There
// 2^n is a normal number, so the two exact power-of-two factors of the
// specification collapse into one multiply with the same single rounding.
// -h = (-silu(g)) * up for two elements, from ng = -g; bit for bit the
// specification's -(silu(g) * up), because negation is exact and every
// rounding used here is symmetric.  Differences of form, all giving the same
// bits:
//  * the exponent x = -g is clamped only below, at -87: below -17 every clamp
//    gives d = 1 exactly (e^-17 is under half an ulp of 1), so -87 reproduces
//    the specification's -104, and it keeps 2^n a normal number, so the two
//    exact power-of-two factors collapse into one multiply with the same
//    single rounding.  Above 80 (g < -80) the value is discarded for +0.
//  * n = rint(t) is (t + 1.5 * 2^23) - 1.5 * 2^23: for |t| < 2^22 the sum lies
//    in [2^23, 2^24), where the spacing is 1, so it rounds t to an integer
//    with ties to even (1.5 * 2^23 is even); the integer sits in the sum's
//    low mantissa bits, from which -2^n is built.
//  * the steps carry nd = -d = -1 + (-e^x); the seed 0x7EF311C7 - bits(d) is
//    0xFEF311C7 - bits(nd) (mod 2^32), and the Newton steps use -d as is.
__device__ __forceinline__ float2 neg_swiglu_f32x2(float2 ng, float2 up) {
    const float2 x = make_float2(fmaxf(ng.x, -87.0f), fmaxf(ng.y, -87.0f));
    const float2 t = __fmul2_rn(x, f2(0x1.715476p+0f));
    const float2 big = __fadd2_rn(t, f2(0x1.8p+23f));
    const float2 n = __fadd2_rn(big, f2(-0x1.8p+23f));
    float2 r = __ffma2_rn(n, f2(-0x1.62e4p-1f), x);
    r = __ffma2_rn(n, f2(-0x1.7f7d1cp-20f), r);
    float2 p = f2(0x1.a01a02p-13f);
    p = __ffma2_rn(p, r, f2(0x1.6c16c2p-10f));
    p = __ffma2_rn(p, r, f2(0x1.111112p-7f));
    p = __ffma2_rn(p, r, f2(0x1.555556p-5f));
    p = __ffma2_rn(p, r, f2(0x1.555556p-3f));
    p = __ffma2_rn(p, r, f2(0.5f));
    p = __ffma2_rn(p, r, f2(1.0f));
    p = __ffma2_rn(p, r, f2(1.0f));
    // -2^n: exponent field n + 127 = bits(big) - bits(1.5 * 2^23) + 127, sign set
    const uint32_t c = ((127u - 0x4B400000u) << 23) | 0x80000000u;
    const float2 m2n = make_float2(__uint_as_float(__float_as_uint(big.x) * 0x800000u + c),
                                   __uint_as_float(__float_as_uint(big.y) * 0x800000u + c));
    const float2 nd = __fadd2_rn(f2(-1.0f), __fmul2_rn(p, m2n));  // -(1 + e^x)
    float2 y = make_float2(__uint_as_float(0xFEF311C7u - __float_as_uint(nd.x)),
                           __uint_as_float(0xFEF311C7u - __float_as_uint(nd.y)));
#pragma unroll
    for (int i = 0; i < 3; ++i) y = __ffma2_rn(__ffma2_rn(nd, y, f2(1.0f)), y, y);
    float2 ns = __fmul2_rn(ng, y);  // -silu(g)
    if (ng.x > 80.0f) ns.x = 0.0f;  // -(g * 0) for g < -80
    if (ng.y > 80.0f) ns.y = 0.0f;
    return __fmul2_rn(ns, up);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Work item t -> row t % M, groups 2 (t / M) and 2 (t / M) + 1.
__global__ void __launch_bounds__(kSwThreads, kSwCtasPerSm)
swiglu_quant_kernel(const uint16_t *__restrict__ g, const uint16_t *__restrict__ u, int64_t ld,
                    int64_t M, int64_t F, uint8_t *__restrict__ q, float *__restrict__ s) {
    jet::griddep_launch_dependents();
    jet::griddep_wait();
    const int lane = threadIdx.x & 31, half = lane >> 4, j = lane & 15;
    const int64_t nfb = F / 128, npairs = (nfb + 1) / 2;
    const int64_t warps = (int64_t)gridDim.x * (kSwThreads / 32);
    // Item t = (pair p, row m) with t = p * M + m; the walk t += warps is
    // kept as (p, m) advanced by (warps / M, warps % M), one division here.
    const int64_t t0 = (int64_t)blockIdx.x * (kSwThreads / 32) + (threadIdx.x >> 5);
    const int64_t dp = warps / M, dm = warps % M;
    int64_t p = t0 / M, m = t0 % M;
    auto advance = [&](int64_t &p_, int64_t &m_) {
        p_ += dp;
        m_ += dm;
        if (m_ >= M) {
            m_ -= M;
            ++p_;
        }
    };
    auto load = [&](int64_t p_, int64_t m_, uint4 &gv, uint4 &uv) {
        const int64_t fb_ = 2 * p_ + half;
        if (p_ < npairs && fb_ < nfb) {
            const int64_t at = m_ * ld + fb_ * 128 + 8 * j;
            gv = ld_stream16(g + at);
            uv = ld_stream16(u + at);
        }
    };
    uint4 gc = make_uint4(0, 0, 0, 0), uc = gc;
    load(p, m, gc, uc);
    while (p < npairs) {
        const int64_t fb = 2 * p + half;
        const bool ok = fb < nfb;
        // the next item's loads go out before this item's arithmetic
        int64_t p2 = p, m2 = m;
        advance(p2, m2);
        uint4 gn = make_uint4(0, 0, 0, 0), un = gn;
        load(p2, m2, gn, un);
        const uint32_t gw[4] = {gc.x, gc.y, gc.z, gc.w}, uw[4] = {uc.x, uc.y, uc.z, uc.w};
        float nh[8];  // -h, for the division routine
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t ng = gw[i] ^ 0x80008000u;  // -gate
            const float2 v = neg_swiglu_f32x2(make_float2(bf16_lo(ng), bf16_hi(ng)),
                                              make_float2(bf16_lo(uw[i]), bf16_hi(uw[i])));
            nh[2 * i] = v.x;
            nh[2 * i + 1] = v.y;
            amax = max_abs2(amax, v.x, v.y);
        }
        // the group's 16 lanes (a lane out of range holds zeros)
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        if (ok) {
            const float sc = group_scale(amax);
            const Divisor dv = make_divisor(sc);
            uint2 out;
            out.x = encode4(nh, dv);
            out.y = encode4(nh + 4, dv);
            *reinterpret_cast<uint2 *>(q + m * F + fb * 128 + 8 * j) = out;
            if (j == 0) s[fb * M + m] = sc;
        }
        gc = gn;
        uc = un;
        p = p2;
        m = m2;
    }
}

}  // namespace

jet_status jet_swiglu_quant_1x128(const uint16_t *gate, const uint16_t *up, int64_t ld,
                                  int64_t M, int64_t F, uint8_t *q, float *s,
                                  jet_stream_t stream) {
    JET_REQUIRE(M >= 0 && F >= 0 && ld >= F, JET_ERR_SHAPE);
    const bool empty = (M == 0 || F == 0);
    JET_REQUIRE(empty || (gate && up && q && s), JET_ERR_NULL);
    JET_REQUIRE(F % 128 == 0 && M < ((int64_t)1 << 31) && ld < ((int64_t)1 << 40), JET_ERR_SHAPE);
    JET_REQUIRE(ld % 8 == 0 && jet::aligned16(gate) && jet::aligned16(up) && jet::aligned16(q) &&
                    jet::aligned16(s),
                JET_ERR_ALIGN);
    jet::DeviceInfo dev;
    jet_status st = jet::current_device(&dev);
    if (st != JET_OK) return st;
    if (empty) return JET_OK;
    const int64_t items = M * ((F / 128 + 1) / 2);
    const int64_t want = (items + kSwThreads / 32 - 1) / (kSwThreads / 32);
    const int64_t cap = (int64_t)dev.num_sms * kSwCtasPerSm;
    return jet::launch_pdl(swiglu_quant_kernel, dim3((unsigned)(want < cap ? want : cap)),
                           dim3(kSwThreads), 0, jet::as_stream(stream), gate, up, ld, M, F, q, s);
}
