// RMSNorm with the 1x128 quantization of its output fused: the q/k/v and
// gate/up projections' inputs are written as FP8 codes and scales straight
// from the residual stream, with no BF16 normalised activation in between.
// The pages run fused activation/RMSNorm operators ("Jet-RL ..."
// (gist.science), "Implementierung") and quantize a linear layer's input in
// the operator that produces it ("英伟达破解AI训练效率难题" (163.com), section 五).
//
// Arithmetic (binary32, every step one IEEE operation with round-to-nearest):
//   sum of squares of a row: lane l of the row's warp adds, in order, the
//     squares of the elements 8 (32 j + l) + t, j = 0, 1, ..., t = 0 .. 7
//     (fused multiply-adds: the square of a BF16 value is exact, so each is
//     one rounding of the addition), then five butterfly levels
//     acc += shfl_xor(acc, d), d = 16, 8, 4, 2, 1 (equal in every lane);
//   ms = ss / K, v = ms + eps, r = 1 / sqrt(v) (IEEE division and square
//     root; r = 0 when v == 0);
//   y = (x * r) * g, then the 1x128 group rule of quant_rule.cuh on the
//     binary32 y.  The products run on -r, giving -y bit for bit (negation is
//     exact and the roundings symmetric), the form the division wants.
//
// One warp per row; lane l holds the 16-byte chunks 32 j + l of the row, so a
// 128-wide group is chunk 16 g .. 16 g + 15: for each j, lanes 0-15 hold group
// 2 j and lanes 16-31 group 2 j + 1.  The row is read twice, the second time
// from L1 or L2 (HBM sees it once).  Measured alternatives, both slower on
// 16384 x 4096: keeping the row in registers between the passes (the
// compiler spilled), and staging each row in shared memory by a bulk copy,
// double buffered per warp (at most 16 warps per SM fit: 2390 GB/s against
// 3190 GB/s for this kernel).
#include <cuda_bf16.h>

#include "jet_common.cuh"
#include "quant_rule.cuh"

namespace {

constexpr int kRnThreads = 256;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// acc += square of each of the 8 BF16 values of a chunk, in order.
__device__ __forceinline__ float add_squares(float acc, const uint4 &c) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = bf16_lo(w[i]), b = bf16_hi(w[i]);
        acc = __fmaf_rn(a, a, acc);
        acc = __fmaf_rn(b, b, acc);
    }
    return acc;
}

// -y of one chunk: (x * -r) * g, eight values.
__device__ __forceinline__ void neg_y(const uint4 &xc, const uint4 &gc, float nr, float (&ny)[8]) {
    const uint32_t xw[4] = {xc.x, xc.y, xc.z, xc.w}, gw[4] = {gc.x, gc.y, gc.z, gc.w};
    const float2 nr2 = make_float2(nr, nr);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __fmul2_rn(make_float2(bf16_lo(xw[i]), bf16_hi(xw[i])), nr2);
        const float2 v = __fmul2_rn(t, make_float2(bf16_lo(gw[i]), bf16_hi(gw[i])));
        ny[2 * i] = v.x;
        ny[2 * i + 1] = v.y;
    }
}

// Quantize this lane's chunk j of row m (its group is 2 j + half); all lanes
// call it (shuffles), lanes past the row's end with `valid` false.
__device__ __forceinline__ void quant_chunk(const uint4 &xc, const uint4 &gc, float nr, bool valid,
                                            int64_t grp, int64_t m, int64_t M, int64_t K, int lane,
                                            uint8_t *__restrict__ q, float *__restrict__ s) {
    float ny[8];
    neg_y(xc, gc, nr, ny);
    float amax = max_abs2(0.0f, ny[0], ny[1]);
    amax = max_abs2(amax, ny[2], ny[3]);
    amax = max_abs2(amax, ny[4], ny[5]);
    amax = max_abs2(amax, ny[6], ny[7]);
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (valid) {
        const float sc = group_scale(amax);
        const Divisor dv = make_divisor(sc);
        uint2 out;
        out.x = encode4(ny, dv);
        out.y = encode4(ny + 4, dv);
        *reinterpret_cast<uint2 *>(q + m * K + grp * 128 + 8 * (lane & 15)) = out;
        if ((lane & 15) == 0) s[grp * M + m] = sc;
    }
}

__device__ __forceinline__ float rms_factor(float acc, int64_t K, float eps) {
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, d));
    const float ms = __fdiv_rn(acc, (float)K);
    const float v = __fadd_rn(ms, eps);
    return v == 0.0f ? 0.0f : __fdiv_rn(1.0f, __fsqrt_rn(v));
}

// Persistent warps, one row at a time: the sum of squares in a first pass
// over the row, the quantization in a second pass whose loads hit L1 or L2
// (the row was just read); both passes issue their loads kRnBatch chunks per
// lane at a time, so that a warp has kRnBatch x 512 bytes in flight.
constexpr int kRnBatch = 4;

__global__ void __launch_bounds__(kRnThreads)
rmsnorm_quant_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ g, int64_t M,
                     int64_t K, float eps, uint8_t *__restrict__ q, float *__restrict__ s) {
    jet::griddep_launch_dependents();
    jet::griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t nchunks = K / 8;
    const int64_t nj = (nchunks + 31) / 32;
    const int64_t warps = (int64_t)gridDim.x * (kRnThreads / 32);
    const uint4 zero = make_uint4(0, 0, 0, 0);
    const uint4 *gain = reinterpret_cast<const uint4 *>(g);
    for (int64_t m = (int64_t)blockIdx.x * (kRnThreads / 32) + (threadIdx.x >> 5); m < M;
         m += warps) {
        const uint4 *row = reinterpret_cast<const uint4 *>(x + m * K);
        float acc = 0.0f;
        for (int64_t j = 0; j < nj; j += kRnBatch) {
            uint4 c[kRnBatch];
#pragma unroll
            for (int u = 0; u < kRnBatch; ++u) {
                const int64_t ci = 32 * (j + u) + lane;
                c[u] = ci < nchunks ? row[ci] : zero;
            }
#pragma unroll
            for (int u = 0; u < kRnBatch; ++u) acc = add_squares(acc, c[u]);
        }
        const float nr = -rms_factor(acc, K, eps);
        for (int64_t j = 0; j < nj; j += kRnBatch) {
            uint4 xc[kRnBatch], gc[kRnBatch];
#pragma unroll
            for (int u = 0; u < kRnBatch; ++u) {
                const int64_t ci = 32 * (j + u) + lane;
                const bool ok = ci < nchunks;
                xc[u] = ok ? row[ci] : zero;
                gc[u] = ok ? gain[ci] : zero;
            }
#pragma unroll
            for (int u = 0; u < kRnBatch; ++u) {
                if (j + u >= nj) break;  // warp-uniform
                const int64_t ci = 32 * (j + u) + lane;
                quant_chunk(xc[u], gc[u], nr, ci < nchunks, 2 * (j + u) + (lane >> 4), m, M, K,
                            lane, q, s);
            }
        }
    }
}

// Few rows (decode: fewer rows than SMs): one CTA per row.  Its 8 warps load
// the row into shared memory in one round trip, warp 0 forms the sum of
// squares from there in the order above, and the 8 warps then quantize the
// row's chunks j = w, w + 8, ... (the same group arithmetic) - so a row no
// longer costs one warp's whole dependent chain.  Rows of at most
// kRnRowCtaMaxK elements (the row's BF16 in dynamic shared memory).
constexpr int64_t kRnRowCtaMaxK = 32768;

__global__ void __launch_bounds__(kRnThreads)
rmsnorm_quant_row_cta_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ g,
                             int64_t M, int64_t K, float eps, uint8_t *__restrict__ q,
                             float *__restrict__ s) {
    extern __shared__ uint4 rowbuf[];  // the row's K / 8 chunks of 8 BF16
    __shared__ float nr_sh;
    jet::griddep_launch_dependents();
    jet::griddep_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t nchunks = K / 8;
    const int64_t nj = (nchunks + 31) / 32;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    const uint4 *gain = reinterpret_cast<const uint4 *>(g);
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        const uint4 *row = reinterpret_cast<const uint4 *>(x + m * K);
        for (int64_t ci = threadIdx.x; ci < nchunks; ci += kRnThreads) rowbuf[ci] = row[ci];
        __syncthreads();
        if (warp == 0) {
            float acc = 0.0f;
            for (int64_t j = 0; j < nj; ++j) {
                const int64_t ci = 32 * j + lane;
                acc = add_squares(acc, ci < nchunks ? rowbuf[ci] : zero);
            }
            const float nr = -rms_factor(acc, K, eps);
            if (lane == 0) nr_sh = nr;
        }
        __syncthreads();
        const float nr = nr_sh;
        for (int64_t j = warp; j < nj; j += kRnThreads / 32) {  // warp-uniform
            const int64_t ci = 32 * j + lane;
            const bool ok = ci < nchunks;
            quant_chunk(ok ? rowbuf[ci] : zero, ok ? gain[ci] : zero, nr, ok,
                        2 * j + (lane >> 4), m, M, K, lane, q, s);
        }
        __syncthreads();  // the next row overwrites rowbuf and nr_sh
    }
}

}  // namespace

jet_status jet_rmsnorm_quant_1x128(const uint16_t *x, const uint16_t *g, int64_t M, int64_t K,
                                   float eps, uint8_t *q, float *s, jet_stream_t stream) {
    JET_REQUIRE(M >= 0 && K >= 0, JET_ERR_SHAPE);
    const bool empty = (M == 0 || K == 0);
    JET_REQUIRE(empty || (x && g && q && s), JET_ERR_NULL);
    JET_REQUIRE(K % 128 == 0 && M < ((int64_t)1 << 31) && K < ((int64_t)1 << 24) &&
                    eps >= 0.0f && eps <= 3.0e38f,
                JET_ERR_SHAPE);
    JET_REQUIRE(jet::aligned16(x) && jet::aligned16(g) && jet::aligned16(q) && jet::aligned16(s),
                JET_ERR_ALIGN);
    jet::DeviceInfo dev;
    jet_status st = jet::current_device(&dev);
    if (st != JET_OK) return st;
    if (empty) return JET_OK;
    if (M <= 2 * (int64_t)dev.num_sms && K <= kRnRowCtaMaxK) {
        static bool attr_set[64] = {};
        if (!attr_set[dev.ordinal]) {
            if (cudaFuncSetAttribute(rmsnorm_quant_row_cta_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(kRnRowCtaMaxK * 2)) != cudaSuccess) {
                cudaGetLastError();
                return JET_ERR_CUDA;
            }
            attr_set[dev.ordinal] = true;
        }
        return jet::launch_pdl(rmsnorm_quant_row_cta_kernel, dim3((unsigned)M), dim3(kRnThreads),
                               (size_t)K * 2, jet::as_stream(stream), x, g, M, K, eps, q, s);
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rmsnorm_quant_kernel, kRnThreads,
                                                      0) != cudaSuccess ||
        per_sm < 1) {
        cudaGetLastError();
        per_sm = 1;
    }
    const int64_t want = (M + kRnThreads / 32 - 1) / (kRnThreads / 32);
    const int64_t cap = (int64_t)dev.num_sms * per_sm;
    return jet::launch_pdl(rmsnorm_quant_kernel, dim3((unsigned)(want < cap ? want : cap)),
                           dim3(kRnThreads), 0, jet::as_stream(stream), x, g, M, K, eps, q, s);
}
