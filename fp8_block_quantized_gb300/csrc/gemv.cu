// Forward product Y = X W^T for a handful of tokens (decode, M <= 4), on
// CUDA cores.  With so few rows of X the product streams the weight codes
// once and does M multiply-adds per weight byte: it is bound by HBM, not by
// any contraction, so the tensor-core kernel's tile set-up, TMEM hand-off and
// split reduction are pure overhead here.  Same arithmetic as the GEMM
// ("Jet-RL ..." gist.science summary, "Quantisierungsschema"; scales of the
// nmedialink page's quantization table):
//   Y[m][n] = sum_kb sx[kb][m] * sw[n/128][kb] * sum_{k in kb} D4(qx[m][k]) D4(qw[n][k])
// Each product of two E4M3 values is exact in FP32; the 16 products of one
// lane and group add up in FP32 (fma.rn.f32.f16 on the exact half-precision
// forms of the codes), are scaled by the group's sx * sw and accumulated in
// FP32; lanes, then warps, are summed in a fixed order (deterministic).
//
// Persistent CTAs (two per SM, one for 3-4 tokens) of 8 warps walk blocks of 8 consecutive weight
// rows (inside one 128-row scale block); warp w takes the 512-wide K chunks
// w, w+8, ... of a row block, lane l the 16 codes at 16l of a chunk (all in
// one 128-wide scale group), so each warp load of a weight row is 512
// contiguous bytes.  A warp's next work item (the next chunk, or the first
// chunk of its next row block) has its 8 rows' codes loaded into registers
// before the current item is computed, so 4 KB per warp stay in flight.
#include <cuda_bf16.h>

#include "jet_common.cuh"
#include "stream_ld.cuh"

namespace {

constexpr int kGemvRows = 8;
constexpr int kGemvThreads = 256;
// two CTAs per SM with up to 2 tokens; one with 3-4 (their accumulators and
// the converted token codes need the registers)
template <int MT>
constexpr int gemv_ctas_per_sm() { return MT <= 2 ? 2 : 1; }

// Four E4M3 codes -> two f16x2 words (exact), lowest code in the low half.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t four, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(four));
}

// 16 codes (one 16-byte load) -> 8 f16x2 words.
__device__ __forceinline__ void unpack16(const uint4 &v, uint32_t (&h)[8]) {
    e4m3x4_to_f16x4(v.x, h[0], h[1]);
    e4m3x4_to_f16x4(v.y, h[2], h[3]);
    e4m3x4_to_f16x4(v.z, h[4], h[5]);
    e4m3x4_to_f16x4(v.w, h[6], h[7]);
}

// sum of the 16 products w_j * x_j, FP32 accumulation in two chains
__device__ __forceinline__ float dot16(const uint32_t (&w)[8], const uint32_t (&x)[8]) {
    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
            "mov.b32 {wl, wh}, %2;\n\t"
            "mov.b32 {xl, xh}, %3;\n\t"
            "fma.rn.f32.f16 %0, wl, xl, %0;\n\t"
            "fma.rn.f32.f16 %1, wh, xh, %1;\n\t}"
            : "+f"(a0), "+f"(a1)
            : "r"(w[j]), "r"(x[j]));
    return a0 + a1;
}

template <int MT>
__global__ void __launch_bounds__(kGemvThreads, gemv_ctas_per_sm<MT>())
gemv_fp8_kernel(const uint8_t *__restrict__ qx, const float *__restrict__ sx,
                const uint8_t *__restrict__ qw, const float *__restrict__ sw, int64_t N,
                int64_t K, uint16_t *__restrict__ y) {
    __shared__ float red[kGemvThreads / 32][kGemvRows][MT];
    jet::griddep_launch_dependents();
    jet::griddep_wait();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t nkb = K / 128;
    // K is a multiple of 128, not always of 512: the last chunk may be 128,
    // 256 or 384 codes wide, taken by its first 8, 16 or 24 lanes.
    const int64_t nsteps = (K + 511) / 512;
    const int64_t nblocks = N / kGemvRows;
    // This warp's work items, in order: row blocks rb = blockIdx.x, +gridDim.x,
    // ...; within a row block the chunks c = w, w + 8, ...  The next item's
    // weight codes are loaded before the current item is computed.
    const int64_t per_rb = w < nsteps ? (nsteps - 1 - w) / (kGemvThreads / 32) + 1 : 0;
    int64_t rb = blockIdx.x, j = 0;  // current item: row block rb, its j-th chunk
    auto load = [&](int64_t rb_, int64_t j_, uint4 (&wr)[kGemvRows]) {
        const int64_t k0 = (w + j_ * (kGemvThreads / 32)) * 512 + 16 * lane;
        if (rb_ < nblocks && j_ < per_rb && k0 < K) {
#pragma unroll
            for (int r = 0; r < kGemvRows; ++r)
                wr[r] = ld_stream16(qw + (rb_ * kGemvRows + r) * K + k0);
        }
    };
    uint4 cur[kGemvRows], nxt[kGemvRows];
    load(rb, j, cur);
    float acc[kGemvRows][MT];
#pragma unroll
    for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = 0.0f;
    while (rb < nblocks) {
        // next item
        int64_t rb2 = rb, j2 = j + 1;
        if (j2 >= per_rb) {
            rb2 = rb + gridDim.x;
            j2 = 0;
        }
        load(rb2, j2, nxt);
        if (j < per_rb) {
            const int64_t k0 = (w + j * (kGemvThreads / 32)) * 512 + 16 * lane;
            if (k0 < K) {
                const int64_t kb = k0 / 128;
                const float swv = sw[(rb * kGemvRows / 128) * nkb + kb];
                uint32_t xh[MT][8];
                float s[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    unpack16(*reinterpret_cast<const uint4 *>(qx + m * K + k0), xh[m]);
                    s[m] = sx[kb * MT + m] * swv;
                }
#pragma unroll
                for (int r = 0; r < kGemvRows; ++r) {
                    uint32_t wh[8];
                    unpack16(cur[r], wh);
#pragma unroll
                    for (int m = 0; m < MT; ++m)
                        acc[r][m] = fmaf(dot16(wh, xh[m]), s[m], acc[r][m]);
                }
            }
        }
        if (j2 == 0) {
            // row block done: lanes, then warps, in a fixed order
#pragma unroll
            for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float v = acc[r][m];
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1)
                        v += __shfl_xor_sync(0xffffffffu, v, off);
                    if (lane == 0) red[w][r][m] = v;
                    acc[r][m] = 0.0f;
                }
            __syncthreads();
            if (threadIdx.x < kGemvRows * MT) {
                const int r = threadIdx.x / MT, m = threadIdx.x % MT;
                float v = red[0][r][m];
#pragma unroll
                for (int i = 1; i < kGemvThreads / 32; ++i) v += red[i][r][m];
                __nv_bfloat16 b = __float2bfloat16_rn(v);
                y[m * N + rb * kGemvRows + r] = *reinterpret_cast<uint16_t *>(&b);
            }
            __syncthreads();
        }
        rb = rb2;
        j = j2;
#pragma unroll
        for (int r = 0; r < kGemvRows; ++r) cur[r] = nxt[r];
    }
}

template <int MT>
jet_status launch_gemv(const uint8_t *qx, const float *sx, const uint8_t *qw, const float *sw,
                       int64_t N, int64_t K, uint16_t *y, int num_sms, cudaStream_t stream) {
    const int64_t blocks = N / kGemvRows, cap = (int64_t)num_sms * gemv_ctas_per_sm<MT>();
    return jet::launch_pdl(gemv_fp8_kernel<MT>, dim3((unsigned)(blocks < cap ? blocks : cap)),
                           dim3(kGemvThreads), 0, stream, qx, sx, qw, sw, N, K, y);
}

}  // namespace

// Forward product for 1 <= M <= 4 tokens; arguments validated by the caller
// (N, K multiples of 128, K > 0, pointers 16-byte aligned).
jet_status jet_gemv_fp8_fwd(const uint8_t *qx, const float *sx, const uint8_t *qw,
                            const float *sw, int64_t M, int64_t N, int64_t K, uint16_t *y,
                            int num_sms, cudaStream_t stream) {
    switch (M) {
    case 1: return launch_gemv<1>(qx, sx, qw, sw, N, K, y, num_sms, stream);
    case 2: return launch_gemv<2>(qx, sx, qw, sw, N, K, y, num_sms, stream);
    case 3: return launch_gemv<3>(qx, sx, qw, sw, N, K, y, num_sms, stream);
    case 4: return launch_gemv<4>(qx, sx, qw, sw, N, K, y, num_sms, stream);
    default: return JET_ERR_SHAPE;
    }
}
