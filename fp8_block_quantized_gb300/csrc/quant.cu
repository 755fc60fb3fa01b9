// Quantization kernels: 1x128 (activations / output gradients), 128x128
// (weights) and the fused transpose + 128x1 re-quantization for WGrad.
//
// Group rule (quantization table of "NVIDIA强化学习加速实操：10分钟提升2倍训练效率",
// section "为什么FP8适配线性层？": E4M3 codes, FP32 scale per group):
//   amax = max |v|, s = amax / 448 (IEEE division, s = 1 if amax == 0),
//   q = cvt.rn.satfinite.e4m3(fl32(v / s)).
// Every kernel is a single pass over HBM: 16-byte loads, the group's amax by
// warp shuffles (and shared memory for 128x128 blocks), the IEEE divide and
// the saturating E4M3 conversion, 8- or 16-byte stores.
#include <cuda_fp8.h>

#include "jet_common.cuh"

namespace {

__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Two E4M3 codes, `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
    __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
    return __half2float(__half(h));
}

__device__ __forceinline__ float group_scale(float amax) {
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
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
__device__ __forceinline__ uint2 encode8(const float f[8], float s) {
    uint2 r;
    r.x = e4m3x2(__fdiv_rn(f[0], s), __fdiv_rn(f[1], s)) |
          (e4m3x2(__fdiv_rn(f[2], s), __fdiv_rn(f[3], s)) << 16);
    r.y = e4m3x2(__fdiv_rn(f[4], s), __fdiv_rn(f[5], s)) |
          (e4m3x2(__fdiv_rn(f[6], s), __fdiv_rn(f[7], s)) << 16);
    return r;
}

// ------------------------------------------------------------------ 1x128 --
// CTA = 256 threads = 16 teams of 16 lanes; a team owns one 1x128 group at a
// time (16 lanes x 8 BF16).  A CTA covers 64 rows of one K-block, four groups
// per team, all four 16-byte loads issued before any arithmetic.
constexpr int kActRowsPerCta = 64;

__global__ void __launch_bounds__(256)
quant_act_1x128_kernel(const uint16_t *__restrict__ x, int64_t M, int64_t K,
                       uint8_t *__restrict__ q, float *__restrict__ s) {
    const int team = threadIdx.x >> 4;
    const int tl = threadIdx.x & 15;
    const int64_t kb = blockIdx.y;
    const int64_t m0 = (int64_t)blockIdx.x * kActRowsPerCta + team;
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
        if (m < M) {
            *reinterpret_cast<uint2 *>(q + m * K + col) = encode8(f, sc);
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
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        float f[8];
        unpack8(v[p], f);
        *reinterpret_cast<uint2 *>(q + (row0 + 16 * p) * K + col) = encode8(f, sc);
    }
    if (threadIdx.x == 0) s[nb * (K / 128) + kb] = sc;
    (void)N;
}

// ------------------------------------------------------------------ 128x1 --
// One CTA per (128 tokens x 128 columns) tile.  Phase 1 stages the codes in
// shared memory with 16-byte loads; phase 2 gives each thread one column and
// 64 tokens: dequantize v = fl32(D4(q) * s_row), column amax over the 128
// tokens (two half-columns meet in shared memory), re-quantize, and write the
// transposed codes as 16-byte stores (one contiguous 64-byte run per thread).
__global__ void __launch_bounds__(256)
requant_128x1_kernel(const uint8_t *__restrict__ q, const float *__restrict__ s,
                     int64_t M, int64_t K, uint8_t *__restrict__ qT,
                     float *__restrict__ sT) {
    __shared__ __align__(16) uint8_t tile[128][128];
    __shared__ float srow[128];
    __shared__ float half_max[2][128];
    const int64_t kb = blockIdx.x, mb = blockIdx.y;
    const int t = threadIdx.x;

#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const int row = (t >> 3) + 32 * p, chunk = t & 7;
        *reinterpret_cast<uint4 *>(&tile[row][chunk * 16]) =
            ld_stream16(q + (mb * 128 + row) * K + kb * 128 + chunk * 16);
    }
    if (t < 128) srow[t] = s[kb * M + mb * 128 + t];
    __syncthreads();

    const int k = t & 127, h = t >> 7;
    float v[64];
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 64; ++i) {
        const int m = h * 64 + i;
        v[i] = e4m3_to_f32(tile[m][k]) * srow[m];
        a = fmaxf(a, fabsf(v[i]));
    }
    half_max[h][k] = a;
    __syncthreads();
    a = fmaxf(half_max[0][k], half_max[1][k]);
    const float sc = group_scale(a);

    uint8_t *dst = qT + (kb * 128 + k) * M + mb * 128 + h * 64;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t w4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = c * 16 + j * 4;
            w4[j] = e4m3x2(__fdiv_rn(v[i], sc), __fdiv_rn(v[i + 1], sc)) |
                    (e4m3x2(__fdiv_rn(v[i + 2], sc), __fdiv_rn(v[i + 3], sc)) << 16);
        }
        *reinterpret_cast<uint4 *>(dst + c * 16) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
    if (h == 0) sT[mb * K + kb * 128 + k] = sc;
}

}  // namespace

extern "C" {

jet_status jet_quant_act_1x128(const uint16_t *x, int64_t M, int64_t K, uint8_t *q,
                               float *s, jet_stream_t stream) {
    JET_REQUIRE(M >= 0 && K >= 0, JET_ERR_SHAPE);
    const bool empty = (M == 0 || K == 0);
    JET_REQUIRE(empty || (x && q && s), JET_ERR_NULL);
    JET_REQUIRE(K % 128 == 0 && K / 128 <= 65535, JET_ERR_SHAPE);
    JET_REQUIRE(jet::aligned16(x) && jet::aligned16(q) && jet::aligned16(s), JET_ERR_ALIGN);
    jet::DeviceInfo dev;
    jet_status st = jet::current_device(&dev);
    if (st != JET_OK) return st;
    if (empty) return JET_OK;
    dim3 grid((unsigned)((M + kActRowsPerCta - 1) / kActRowsPerCta), (unsigned)(K / 128));
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
