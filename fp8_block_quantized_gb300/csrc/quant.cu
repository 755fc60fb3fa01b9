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
#include <cuda.h>
#include <cuda_fp8.h>

#include <mutex>

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

// All three kernels stage their input tile in shared memory with one 2D TMA
// load (box = the whole tile, no swizzle; rows past the end of the tensor are
// zero-filled) completing on one mbarrier, then compute from shared memory.
// Loads in flight cost no registers, so several tiles are in flight per SM.
using jet::ptx::bulk_g2s;
using jet::ptx::tma_load_2d;
using jet::ptx::mbar_arrive_expect_tx;
using jet::ptx::mbar_init;
using jet::ptx::mbar_wait;
using jet::ptx::smem_u32;

// Inputs are read once: a plain (evict-normal) policy value for the hinted
// TMA load.  createpolicy with fraction 0 yields the default policy.
#define kStreamPolicy jet::ptx::policy_evict_first()

__device__ __forceinline__ void stage_init(uint64_t *bar) {
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        jet::ptx::fence_mbar_init();
    }
    __syncthreads();
}

// ------------------------------------------------------------------ 1x128 --
// CTA = 256 threads = 16 teams of 16 lanes and one tile of 64 rows x one
// K-block (16 KB of BF16, up to eight CTAs per SM).  A team owns one 1x128
// group at a time (16 lanes x 8 BF16 read from shared memory); the group's
// amax by shuffles within the team.  K-blocks are the fast grid index, so
// CTAs running together read whole rows.
constexpr int kActRowsPerCta = 64;

__global__ void __launch_bounds__(256)
quant_act_1x128_kernel(const __grid_constant__ CUtensorMap tmx, int64_t M, int64_t K,
                       uint8_t *__restrict__ q, float *__restrict__ s, unsigned *status) {
    __shared__ __align__(128) uint16_t tile[kActRowsPerCta][128];
    __shared__ uint64_t bar;
    const int team = threadIdx.x >> 4, tl = threadIdx.x & 15;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t kb = blockIdx.x;
    const int64_t mbase = (int64_t)blockIdx.y * kActRowsPerCta;
    const int rows = (int)(M - mbase < kActRowsPerCta ? M - mbase : kActRowsPerCta);
    stage_init(&bar);
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&bar, (uint32_t)sizeof(tile));
        tma_load_2d(smem_u32(&tile[0][0]), &tmx, &bar, (int32_t)(kb * 128), (int32_t)mbase,
                    kStreamPolicy);
    }
    (void)warp;
    (void)lane;
    if (!mbar_wait(&bar, 0, nullptr, status, jet::SITE_QUANT_STAGE)) return;
#pragma unroll
    for (int j = 0; j < kActRowsPerCta / 16; ++j) {
        const int r = team + 16 * j;
        const uint4 v = *reinterpret_cast<const uint4 *>(&tile[r][tl * 8]);
        float f[8];
        unpack8(v, f);
        float a = absmax8(f);
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
        if (r < rows) {
            const float sc = group_scale(a);
            const Divisor d = make_divisor(sc);
            const int64_t m = mbase + r;
            *reinterpret_cast<uint2 *>(q + m * K + kb * 128 + tl * 8) = encode8(f, d);
            if (tl == 0) s[kb * M + m] = sc;
        }
    }
}

// ---------------------------------------------------------------- 128x128 --
// One CTA per 128x128 block (32 KB of BF16 in shared memory, six CTAs per
// SM).  Pass 1: each thread's 64 values -> block amax (shuffles, then
// shared memory).  Pass 2: the same values re-read, quantized, stored.
__global__ void __launch_bounds__(256)
quant_w_128x128_kernel(const __grid_constant__ CUtensorMap tmw, int64_t N, int64_t K,
                       uint8_t *__restrict__ q, float *__restrict__ s, unsigned *status) {
    extern __shared__ __align__(128) uint8_t wsm[];
    uint16_t(*tile)[128] = reinterpret_cast<uint16_t(*)[128]>(wsm);
    __shared__ uint64_t bar;
    __shared__ float warp_max[8];
    const int64_t kb = blockIdx.x, nb = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = threadIdx.x >> 4, tl = threadIdx.x & 15;
    stage_init(&bar);
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&bar, 128u * 256u);
        tma_load_2d(smem_u32(&tile[0][0]), &tmw, &bar, (int32_t)(kb * 128), (int32_t)(nb * 128),
                    kStreamPolicy);
    }
    if (!mbar_wait(&bar, 0, nullptr, status, jet::SITE_QUANT_STAGE)) return;
    float a = 0.0f;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        float f[8];
        unpack8(*reinterpret_cast<const uint4 *>(&tile[r0 + 16 * p][tl * 8]), f);
        a = fmaxf(a, absmax8(f));
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    if (lane == 0) warp_max[warp] = a;
    __syncthreads();
    a = warp_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) a = fmaxf(a, warp_max[i]);
    const float sc = group_scale(a);
    const Divisor d = make_divisor(sc);
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        float f[8];
        unpack8(*reinterpret_cast<const uint4 *>(&tile[r0 + 16 * p][tl * 8]), f);
        *reinterpret_cast<uint2 *>(q + (nb * 128 + r0 + 16 * p) * K + kb * 128 + tl * 8) =
            encode8(f, d);
    }
    if (threadIdx.x == 0) s[nb * (K / 128) + kb] = sc;
    (void)N;
}

// ------------------------------------------------------------------ 128x1 --
// One CTA (8 warps) per (128 tokens x 128 columns) tile: 16 KB of codes and
// the 128 row scales in shared memory (four CTAs per SM at 64 registers).  Lane l of
// warp w owns columns 4l .. 4l+3 and tokens 16w .. 16w+15.  Pass 1 reads its
// 16 words, dequantizes v = fl32(D4(q) * s_row) and reduces the column maxima
// over its tokens; the 8 warps meet in shared memory for the 128-token
// column amax.  Pass 2 re-reads, dequantizes two columns x 8 tokens at a
// time, re-quantizes and writes each column's 8 codes as one 8-byte store
// into the transposed output.
__global__ void __launch_bounds__(256, 4)
requant_128x1_kernel(const __grid_constant__ CUtensorMap tmq, const float *__restrict__ s,
                     int64_t M, int64_t K, uint8_t *__restrict__ qT,
                     float *__restrict__ sT, unsigned *status) {
    __shared__ __align__(128) uint32_t tile[128][32];  // [token][4 codes]
    __shared__ __align__(16) float srow[128];
    __shared__ __align__(16) float col_max[8][128];
    __shared__ uint64_t bar;
    const int64_t kb = blockIdx.x, mb = blockIdx.y;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    stage_init(&bar);
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&bar, 128u * 128u + 512u);
        tma_load_2d(smem_u32(&tile[0][0]), &tmq, &bar, (int32_t)(kb * 128), (int32_t)(mb * 128),
                    kStreamPolicy);
        bulk_g2s(smem_u32(srow), s + kb * M + mb * 128, 512u, &bar);
    }
    if (!mbar_wait(&bar, 0, nullptr, status, jet::SITE_QUANT_STAGE)) return;
    const int t0 = w * 16;

    // pass 1: column maxima of v = fl32(D4(q) * s_row)
    float amax[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t code = tile[t0 + i][lane];
        float d0, d1, d2, d3;
        e4m3x2_to_f32(code, d0, d1);
        e4m3x2_to_f32(code >> 16, d2, d3);
        const float2 sr = make_float2(srow[t0 + i], srow[t0 + i]);
        const float2 v01 = __fmul2_rn(make_float2(d0, d1), sr);
        const float2 v23 = __fmul2_rn(make_float2(d2, d3), sr);
        amax[0] = fmaxf(amax[0], fabsf(v01.x));
        amax[1] = fmaxf(amax[1], fabsf(v01.y));
        amax[2] = fmaxf(amax[2], fabsf(v23.x));
        amax[3] = fmaxf(amax[3], fabsf(v23.y));
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
    for (int c = 0; c < 4; ++c) sc[c] = group_scale(amax[c]);

    // pass 2: two columns x 8 tokens at a time
    const int64_t col = kb * 128 + lane * 4;
    const int64_t m0 = mb * 128 + t0;
#pragma unroll
    for (int cp = 0; cp < 2; ++cp) {
        const Divisor d0 = make_divisor(sc[2 * cp]), d1 = make_divisor(sc[2 * cp + 1]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float va[8], vb[8];  // column 2cp and 2cp+1, tokens 8h .. 8h+7
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int t = t0 + 8 * h + i;
                float x0, x1;
                e4m3x2_to_f32(tile[t][lane] >> (16 * cp), x0, x1);
                const float2 v = __fmul2_rn(make_float2(x0, x1), make_float2(srow[t], srow[t]));
                va[i] = v.x;
                vb[i] = v.y;
            }
            uint32_t oa[2], ob[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float q0, q1, q2, q3;
                qdiv2(va[4 * j + 0], va[4 * j + 1], d0, q0, q1);
                qdiv2(va[4 * j + 2], va[4 * j + 3], d0, q2, q3);
                oa[j] = e4m3x2(q0, q1) | (e4m3x2(q2, q3) << 16);
                qdiv2(vb[4 * j + 0], vb[4 * j + 1], d1, q0, q1);
                qdiv2(vb[4 * j + 2], vb[4 * j + 3], d1, q2, q3);
                ob[j] = e4m3x2(q0, q1) | (e4m3x2(q2, q3) << 16);
            }
            *reinterpret_cast<uint2 *>(qT + (col + 2 * cp) * M + m0 + 8 * h) =
                make_uint2(oa[0], oa[1]);
            *reinterpret_cast<uint2 *>(qT + (col + 2 * cp + 1) * M + m0 + 8 * h) =
                make_uint2(ob[0], ob[1]);
        }
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

constexpr int kWTileBytes = 128 * 128 * 2;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        cudaGetLastError();
    });
    return fn;
}

// Row-major [outer][inner] tensor of 1- or 2-byte elements, box box_outer x
// box_inner, no swizzle, zero fill outside.
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType type, uint32_t esize,
              uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * esize};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, type, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
    CUtensorMap tm;
    if (!make_map(&tm, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)K, (uint64_t)M, 128,
                  kActRowsPerCta))
        return JET_ERR_CUDA;
    dim3 grid((unsigned)(K / 128), (unsigned)((M + kActRowsPerCta - 1) / kActRowsPerCta));
    quant_act_1x128_kernel<<<grid, 256, 0, jet::as_stream(stream)>>>(tm, M, K, q, s,
                                                                     dev.status_word);
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
    static bool attr_set[64] = {};
    if (!attr_set[dev.ordinal]) {
        if (cudaFuncSetAttribute(quant_w_128x128_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kWTileBytes) != cudaSuccess) {
            cudaGetLastError();
            return JET_ERR_CUDA;
        }
        attr_set[dev.ordinal] = true;
    }
    CUtensorMap tm;
    if (!make_map(&tm, w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)K, (uint64_t)N, 128, 128))
        return JET_ERR_CUDA;
    dim3 grid((unsigned)(K / 128), (unsigned)(N / 128));
    quant_w_128x128_kernel<<<grid, 256, kWTileBytes, jet::as_stream(stream)>>>(tm, N, K, q, s,
                                                                               dev.status_word);
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
    CUtensorMap tm;
    if (!make_map(&tm, q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)K, (uint64_t)M, 128, 128))
        return JET_ERR_CUDA;
    dim3 grid((unsigned)(K / 128), (unsigned)(M / 128));
    requant_128x1_kernel<<<grid, 256, 0, jet::as_stream(stream)>>>(tm, s, M, K, qT, sT,
                                                                   dev.status_word);
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
