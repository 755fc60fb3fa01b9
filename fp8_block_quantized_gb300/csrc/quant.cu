// Quantization kernels: 1x128 (activations / output gradients), 128x128
// (weights) and the fused transpose + 128x1 re-quantization for WGrad.
//
// Group rule (quantization table of "NVIDIA强化学习加速实操：10分钟提升2倍训练效率",
// section "为什么FP8适配线性层？": E4M3 codes, FP32 scale per group):
//   amax = max |v|, s = amax / 448 (IEEE division, s = 1 if amax == 0),
//   q = cvt.rn.satfinite.e4m3(fl32(v / s)).
// Every kernel is a single pass over HBM: coalesced 16- or 4-byte loads, the
// group's amax by warp shuffles or shared memory, a correctly rounded divide
// by the group scale (Markstein, below) and the saturating E4M3 conversion,
// 8- or 16-byte stores.
#include <cuda_fp8.h>

#include "jet_common.cuh"
#include "sm100_ptx.cuh"

namespace {


__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_stream4(const void *p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Two E4M3 codes, `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// Two E4M3 codes (low byte first) -> two exact floats.
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t two, float &lo, float &hi) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
    lo = __half2float(__half(__half_raw{h.x}));
    hi = __half2float(__half(__half_raw{h.y}));
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
// rounding boundary, so their codes are the same.  copysign restores the sign
// of zero quotients.  Groups with s < 2^-90 divide with __fdiv_rn.
// ---------------------------------------------------------------------------
struct Divisor {
    float s, ns, y;
    bool fast;
};

__device__ __forceinline__ Divisor make_divisor(float s) {
    Divisor d;
    d.s = s;
    d.ns = -s;
    d.fast = s >= 0x1p-90f;
    d.y = d.fast ? __frcp_rn(s) : 0.0f;
    return d;
}

__device__ __forceinline__ float qdiv(float x, const Divisor &d) {
    if (!d.fast) return __fdiv_rn(x, d.s);
    float q = __fmul_rn(x, d.y);
    float r = __fmaf_rn(q, d.ns, x);
    q = __fmaf_rn(r, d.y, q);
    r = __fmaf_rn(q, d.ns, x);
    q = __fmaf_rn(r, d.y, q);
    return copysignf(q, x);
}

// Two quotients with packed f32x2 arithmetic (same steps as qdiv).
__device__ __forceinline__ void qdiv2(float x0, float x1, const Divisor &d, float &q0, float &q1) {
    if (!d.fast) {
        q0 = __fdiv_rn(x0, d.s);
        q1 = __fdiv_rn(x1, d.s);
        return;
    }
    const float2 x = make_float2(x0, x1), y = make_float2(d.y, d.y);
    const float2 ns = make_float2(d.ns, d.ns);
    float2 q = __fmul2_rn(x, y);
    float2 r = __ffma2_rn(q, ns, x);
    q = __ffma2_rn(r, y, q);
    r = __ffma2_rn(q, ns, x);
    q = __ffma2_rn(r, y, q);
    q0 = copysignf(q.x, x0);
    q1 = copysignf(q.y, x1);
}

// Eight BF16 values (one 16-byte load) -> eight floats.
__device__ __forceinline__ void unpack8(const uint4 &v, float f[8]) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

__device__ __forceinline__ float absmax8(const float f[8]) {
    float a = fabsf(f[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) a = fmaxf(a, fabsf(f[i]));
    return a;
}

// Eight quotients f[i] / s -> eight codes packed little-endian in a uint2.
__device__ __forceinline__ uint2 encode8(const float f[8], const Divisor &d) {
    float q[8];
#pragma unroll
    for (int i = 0; i < 8; i += 2) qdiv2(f[i], f[i + 1], d, q[i], q[i + 1]);
    uint2 r;
    r.x = e4m3x2(q[0], q[1]) | (e4m3x2(q[2], q[3]) << 16);
    r.y = e4m3x2(q[4], q[5]) | (e4m3x2(q[6], q[7]) << 16);
    return r;
}

// ------------------------------------------------------------------ 1x128 --
// CTA = 256 threads = 16 teams of 16 lanes; a team owns one 1x128 group at a
// time (16 lanes x 8 BF16).  A CTA covers 64 rows of one K-block, four groups
// per team, all four 16-byte loads issued before any arithmetic.  K-blocks are
// the fast grid index, so CTAs running together read whole rows.
constexpr int kActRowsPerCta = 64;

__global__ void __launch_bounds__(256)
quant_act_1x128_kernel(const uint16_t *__restrict__ x, int64_t M, int64_t K,
                       uint8_t *__restrict__ q, float *__restrict__ s) {
    const int team = threadIdx.x >> 4;
    const int tl = threadIdx.x & 15;
    const int64_t kb = blockIdx.x;
    const int64_t m0 = (int64_t)blockIdx.y * kActRowsPerCta + team;
    const int64_t col = kb * 128 + tl * 8;

    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t m = m0 + 16 * j;
        v[j] = m < M ? ld_stream16(x + m * K + col) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t m = m0 + 16 * j;
        float f[8];
        unpack8(v[j], f);
        float a = absmax8(f);
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
        const float sc = group_scale(a);
        const Divisor d = make_divisor(sc);
        if (m < M) {
            *reinterpret_cast<uint2 *>(q + m * K + col) = encode8(f, d);
            if (tl == 0) s[kb * M + m] = sc;
        }
    }
}

// ---------------------------------------------------------------- 128x128 --
// One CTA per 128x128 block; each thread holds 64 values (eight 16-byte
// loads); block amax by warp shuffle then shared memory.
__global__ void __launch_bounds__(256)
quant_w_128x128_kernel(const uint16_t *__restrict__ w, int64_t N, int64_t K,
                       uint8_t *__restrict__ q, float *__restrict__ s) {
    __shared__ float warp_max[8];
    const int64_t kb = blockIdx.x, nb = blockIdx.y;
    const int r0 = threadIdx.x >> 4, tl = threadIdx.x & 15;
    const int64_t col = kb * 128 + tl * 8;
    const int64_t row0 = nb * 128 + r0;

    uint4 v[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) v[p] = ld_stream16(w + (row0 + 16 * p) * K + col);
    float a = 0.0f;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        float f[8];
        unpack8(v[p], f);
        a = fmaxf(a, absmax8(f));
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = a;
    __syncthreads();
    a = warp_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) a = fmaxf(a, warp_max[i]);
    const float sc = group_scale(a);
    const Divisor d = make_divisor(sc);
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        float f[8];
        unpack8(v[p], f);
        *reinterpret_cast<uint2 *>(q + (row0 + 16 * p) * K + col) = encode8(f, d);
    }
    if (threadIdx.x == 0) s[nb * (K / 128) + kb] = sc;
    (void)N;
}

// ------------------------------------------------------------------ 128x1 --
// One CTA (8 warps) per (128 tokens x 128 columns) tile.  Lane l of warp w
// owns columns 4l .. 4l+3 and tokens 16w .. 16w+15: it reads its 16 rows as
// 4-byte words (each warp instruction reads one contiguous 128-byte row
// segment), dequantizes v = fl32(D4(q) * s_row), reduces its column maxima
// over its 16 tokens, meets the other 7 warps in shared memory for the
// 128-token column amax, re-quantizes, and writes each column's 16 codes as
// one 16-byte store into the transposed output.
__global__ void __launch_bounds__(256)
requant_128x1_kernel(const uint8_t *__restrict__ q, const float *__restrict__ s,
                     int64_t M, int64_t K, uint8_t *__restrict__ qT,
                     float *__restrict__ sT) {
    __shared__ __align__(16) float col_max[8][128];
    const int64_t kb = blockIdx.x, mb = blockIdx.y;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t m0 = mb * 128 + w * 16;
    const int64_t col = kb * 128 + lane * 4;

    uint32_t code[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) code[i] = ld_stream4(q + (m0 + i) * K + col);
    float srow[16];
    const float4 *s4 = reinterpret_cast<const float4 *>(s + kb * M + m0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 t = __ldg(s4 + i);
        srow[4 * i + 0] = t.x; srow[4 * i + 1] = t.y;
        srow[4 * i + 2] = t.z; srow[4 * i + 3] = t.w;
    }

    float v[4][16];  // [column][token]
    float amax[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float d0, d1, d2, d3;
        e4m3x2_to_f32(code[i], d0, d1);
        e4m3x2_to_f32(code[i] >> 16, d2, d3);
        const float2 sr = make_float2(srow[i], srow[i]);
        const float2 v01 = __fmul2_rn(make_float2(d0, d1), sr);
        const float2 v23 = __fmul2_rn(make_float2(d2, d3), sr);
        v[0][i] = v01.x; v[1][i] = v01.y; v[2][i] = v23.x; v[3][i] = v23.y;
#pragma unroll
        for (int c = 0; c < 4; ++c) amax[c] = fmaxf(amax[c], fabsf(v[c][i]));
    }
    *reinterpret_cast<float4 *>(&col_max[w][lane * 4]) =
        make_float4(amax[0], amax[1], amax[2], amax[3]);
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float4 t = *reinterpret_cast<const float4 *>(&col_max[j][lane * 4]);
        amax[0] = fmaxf(amax[0], t.x); amax[1] = fmaxf(amax[1], t.y);
        amax[2] = fmaxf(amax[2], t.z); amax[3] = fmaxf(amax[3], t.w);
    }
    float sc[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        sc[c] = group_scale(amax[c]);
        const Divisor d = make_divisor(sc[c]);
        uint32_t out[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float q0, q1, q2, q3;
            qdiv2(v[c][4 * j + 0], v[c][4 * j + 1], d, q0, q1);
            qdiv2(v[c][4 * j + 2], v[c][4 * j + 3], d, q2, q3);
            out[j] = e4m3x2(q0, q1) | (e4m3x2(q2, q3) << 16);
        }
        *reinterpret_cast<uint4 *>(qT + (col + c) * M + m0) =
            make_uint4(out[0], out[1], out[2], out[3]);
    }
    if (w == 0)
        *reinterpret_cast<float4 *>(sT + mb * K + col) = make_float4(sc[0], sc[1], sc[2], sc[3]);
}

// Self-test of the division used above: q[i] = x[i] / s[i] through
// make_divisor + qdiv, the same path the quantizers take for a group scale.
__global__ void selftest_quotient_kernel(const float *__restrict__ x, const float *__restrict__ s,
                                         int64_t n, float *__restrict__ q) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        q[i] = qdiv(x[i], make_divisor(s[i]));
}

}  // namespace

extern "C" {

jet_status jet_quant_act_1x128(const uint16_t *x, int64_t M, int64_t K, uint8_t *q,
                               float *s, jet_stream_t stream) {
    JET_REQUIRE(M >= 0 && K >= 0, JET_ERR_SHAPE);
    const bool empty = (M == 0 || K == 0);
    JET_REQUIRE(empty || (x && q && s), JET_ERR_NULL);
    JET_REQUIRE(K % 128 == 0 && (M + kActRowsPerCta - 1) / kActRowsPerCta <= 65535, JET_ERR_SHAPE);
    JET_REQUIRE(jet::aligned16(x) && jet::aligned16(q) && jet::aligned16(s), JET_ERR_ALIGN);
    jet::DeviceInfo dev;
    jet_status st = jet::current_device(&dev);
    if (st != JET_OK) return st;
    if (empty) return JET_OK;
    dim3 grid((unsigned)(K / 128), (unsigned)((M + kActRowsPerCta - 1) / kActRowsPerCta));
    quant_act_1x128_kernel<<<grid, 256, 0, jet::as_stream(stream)>>>(x, M, K, q, s);
    return jet::launch_status();
}

jet_status jet_quant_w_128x128(const uint16_t *w, int64_t N, int64_t K, uint8_t *q,
                               float *s, jet_stream_t stream) {
    JET_REQUIRE(N >= 0 && K >= 0, JET_ERR_SHAPE);
    const bool empty = (N == 0 || K == 0);
    JET_REQUIRE(empty || (w && q && s), JET_ERR_NULL);
    JET_REQUIRE(N % 128 == 0 && K % 128 == 0 && N / 128 <= 65535, JET_ERR_SHAPE);
    JET_REQUIRE(jet::aligned16(w) && jet::aligned16(q) && jet::aligned16(s), JET_ERR_ALIGN);
    jet::DeviceInfo dev;
    jet_status st = jet::current_device(&dev);
    if (st != JET_OK) return st;
    if (empty) return JET_OK;
    dim3 grid((unsigned)(K / 128), (unsigned)(N / 128));
    quant_w_128x128_kernel<<<grid, 256, 0, jet::as_stream(stream)>>>(w, N, K, q, s);
    return jet::launch_status();
}

jet_status jet_requant_128x1(const uint8_t *q, const float *s, int64_t M, int64_t K,
                             uint8_t *qT, float *sT, jet_stream_t stream) {
    JET_REQUIRE(M >= 0 && K >= 0, JET_ERR_SHAPE);
    const bool empty = (M == 0 || K == 0);
    JET_REQUIRE(empty || (q && s && qT && sT), JET_ERR_NULL);
    JET_REQUIRE(M % 128 == 0 && K % 128 == 0 && M / 128 <= 65535, JET_ERR_SHAPE);
    JET_REQUIRE(jet::aligned16(q) && jet::aligned16(s) && jet::aligned16(qT) &&
                    jet::aligned16(sT),
                JET_ERR_ALIGN);
    jet::DeviceInfo dev;
    jet_status st = jet::current_device(&dev);
    if (st != JET_OK) return st;
    if (empty) return JET_OK;
    dim3 grid((unsigned)(K / 128), (unsigned)(M / 128));
    requant_128x1_kernel<<<grid, 256, 0, jet::as_stream(stream)>>>(q, s, M, K, qT, sT);
    return jet::launch_status();
}

}  // extern "C"

extern "C" jet_status jet_selftest_quotient(const float *x, const float *s, int64_t n, float *q,
                                            jet_stream_t stream) {
    JET_REQUIRE(n >= 0, JET_ERR_SHAPE);
    JET_REQUIRE(n == 0 || (x && s && q), JET_ERR_NULL);
    JET_REQUIRE(jet::aligned16(x) && jet::aligned16(s) && jet::aligned16(q), JET_ERR_ALIGN);
    jet::DeviceInfo dev;
    jet_status st = jet::current_device(&dev);
    if (st != JET_OK) return st;
    if (n == 0) return JET_OK;
    const int64_t blocks = (n + 255) / 256;
    selftest_quotient_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0,
                               jet::as_stream(stream)>>>(x, s, n, q);
    return jet::launch_status();
}
