// Quantization kernels: 1x128 (activations / output gradients), 128x128
// (weights) and the fused transpose + 128x1 re-quantization for WGrad.
//
// The group rule (amax, scale, correctly rounded division, E4M3 conversion)
// is in quant_rule.cuh.  Every kernel is a single pass over HBM: TMA tile
// loads into shared memory, the group's amax by warp shuffles and shared
// memory, the division by the group scale and the saturating E4M3
// conversion, 16-byte stores.
#include <cuda.h>
#include <cuda_fp8.h>

#include <mutex>

#include "jet_common.cuh"
#include "quant_rule.cuh"
#include "sm100_ptx.cuh"

namespace {

// Eight BF16 values (one 16-byte load) -> eight negated floats (BF16 is the
// upper half of a binary32; the sign bit is flipped on the way).
__device__ __forceinline__ void unpack8_neg(const uint4 &v, float f[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float((w[i] << 16) + 0x80000000u);
        f[2 * i + 1] = __uint_as_float((w[i] & 0xFFFF0000u) ^ 0x80000000u);
    }
}

// All three kernels stage their input tiles in shared memory by TMA (rows
// past the end of the tensor are zero-filled) completing on an mbarrier, then
// compute from shared memory.  Loads in flight cost no registers.
using jet::ptx::bulk_g2s;
using jet::ptx::tma_load_2d;
using jet::ptx::mbar_arrive_expect_tx;
using jet::ptx::mbar_init;
using jet::ptx::mbar_wait;
using jet::ptx::smem_u32;

// Inputs are read once: they are loaded with the evict-first L2 policy.
#define kStreamPolicy jet::ptx::policy_evict_first()

// 16-byte shared-memory load at a shared-window address.
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// Address of 16-byte chunk `c` (0 .. 7) of row `r` in a box of 128-byte rows
// loaded by TMA with the 128-byte swizzle (the box starts 1024-byte aligned):
// the chunk sits at position c XOR (r mod 8) of its row.
__device__ __forceinline__ uint32_t swz128(uint32_t box, int r, int c) {
    return box + (uint32_t)r * 128u + ((uint32_t)(c ^ (r & 7)) << 4);
}

// The quantizers below are persistent: CTAs walk their tiles with a
// two-stage ring; each tile arrives by TMA loads on the stage's mbarrier and
// the load of the tile after next is issued as soon as the current tile has
// been read into registers, so one load is always in flight per CTA while
// another tile is computed.
using jet::ptx::fence_proxy_async;

// ------------------------------------------------------------------ 1x128 --
// Tile = 64 rows x one K-block (128 BF16 = two 64-column boxes of 128-byte
// rows with the 128-byte swizzle, 16 KB).  Four lanes per 1x128 group, 32
// values each: lane tl of team r holds columns 16tl .. 16tl+15 of each box
// (chunks 2tl and 2tl+1), read one chunk per box and step, so that the eight
// lanes of every quarter-warp touch eight different bank groups (the
// granularity at which 16-byte shared loads are served); the group's amax by
// two shuffles, one scale and reciprocal per group, two 16-byte code stores.
// Tiles are ordered K-block fastest so that CTAs running together read whole
// rows.
constexpr int kActRowsPerCta = 64;
constexpr int kActBoxBytes = kActRowsPerCta * 128;
constexpr int kActTileBytes = 2 * kActBoxBytes;
constexpr int kActCtasPerSm = 4;
constexpr int kActSmemBytes = 2 * kActTileBytes + 1024;

__global__ void __launch_bounds__(256, kActCtasPerSm)
quant_act_1x128_kernel(const __grid_constant__ CUtensorMap tmx, int64_t M, int64_t K,
                       uint8_t *__restrict__ q, float *__restrict__ s, unsigned *status) {
    extern __shared__ uint8_t act_smem[];
    __shared__ uint64_t full[2];
    const uint32_t base = (smem_u32(act_smem) + 1023u) & ~1023u;
    const int row = threadIdx.x >> 2, tl = threadIdx.x & 3;
    const int64_t nkb = K / 128;
    const int64_t ntiles = (M + kActRowsPerCta - 1) / kActRowsPerCta * nkb;
    const int64_t step = gridDim.x;
    if (threadIdx.x == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        jet::ptx::fence_mbar_init();
    }
    __syncthreads();
    jet::griddep_launch_dependents();
    jet::griddep_wait();
    auto issue = [&](int st, int64_t t) {
        const int64_t mb = t / nkb, kb = t - mb * nkb;
        const uint32_t dst = base + st * kActTileBytes;
        mbar_arrive_expect_tx(&full[st], kActTileBytes);
        tma_load_2d(dst, &tmx, &full[st], (int32_t)(kb * 128), (int32_t)(mb * kActRowsPerCta),
                    kStreamPolicy);
        tma_load_2d(dst + kActBoxBytes, &tmx, &full[st], (int32_t)(kb * 128 + 64),
                    (int32_t)(mb * kActRowsPerCta), kStreamPolicy);
    };
    int64_t issued = 0;
    if (threadIdx.x == 0)
        for (int j = 0; j < 2 && blockIdx.x + j * step < ntiles; ++j, ++issued)
            issue(j, blockIdx.x + j * step);
    uint32_t it = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < ntiles; t += step, ++it) {
        const int st = it & 1;
        // A wait that gave up is agreed on at the barrier below, before any
        // global write; until then the (possibly incomplete) stage is only read.
        ok = mbar_wait(&full[st], (it >> 1) & 1u, nullptr, status, jet::SITE_QUANT_STAGE);
        const uint32_t tile = base + st * kActTileBytes;
        float f[32];  // -x: columns 16tl .. 16tl+15, then 64+16tl .. 64+16tl+15
#pragma unroll
        for (int k = 0; k < 4; ++k)
            unpack8_neg(lds128(swz128(tile + (k >> 1) * kActBoxBytes, row, 2 * tl + (k & 1))),
                        f + 8 * k);
        if (__syncthreads_or(!ok)) {
            ok = false;
            break;
        }
        if (threadIdx.x == 0 && t + 2 * step < ntiles) {
            fence_proxy_async();
            issue(st, t + 2 * step);
            ++issued;
        }
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; i += 2) a = max_abs2(a, f[i], f[i + 1]);
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        const int64_t mb = t / nkb, kb = t - mb * nkb;
        const int64_t m = mb * kActRowsPerCta + row;
        if (m < M) {
            const float sc = group_scale(a);
            const Divisor d = make_divisor(sc);
            uint32_t w[8];
            if (d.fast) {
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = encode4_fast(f + 4 * i, d);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = encode4(f + 4 * i, d);
            }
            uint8_t *dst = q + m * K + kb * 128 + tl * 16;
            *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4 *>(dst + 64) = make_uint4(w[4], w[5], w[6], w[7]);
            if (tl == 0) s[kb * M + m] = sc;
        }
    }
    // After a time-out, loads still in flight must land before the CTA exits.
    if (!ok && threadIdx.x == 0)
        for (int64_t j = it; j < issued; ++j)
            mbar_wait(&full[j & 1], (uint32_t)(j >> 1) & 1u, nullptr, status,
                      jet::SITE_QUANT_STAGE);
}

// ---------------------------------------------------------------- 128x128 --
// Tile = one 128x128 block (two 64-column boxes, 128-byte swizzle, 32 KB).
// Thread i holds row i/2, columns 64h .. 64h+63 (h = i%2, one box row) in
// registers, reading chunk k XOR 4h at step k so that the two halves of a
// quarter-warp fall on different bank groups; the block amax by shuffles and
// a shared-memory exchange between the 8 warps, one scale and reciprocal per
// block, 64 contiguous codes per thread.
constexpr int kWBoxBytes = 128 * 128;
constexpr int kWTileBytes = 2 * kWBoxBytes;
constexpr int kWCtasPerSm = 2;
constexpr int kWSmemBytes = 2 * kWTileBytes + 1024;

__global__ void __launch_bounds__(256, kWCtasPerSm)
quant_w_128x128_kernel(const __grid_constant__ CUtensorMap tmw, int64_t N, int64_t K,
                       uint8_t *__restrict__ q, float *__restrict__ s, unsigned *status) {
    extern __shared__ uint8_t w_smem[];
    __shared__ uint64_t full[2];
    __shared__ float warp_max[2][8];
    const uint32_t base = (smem_u32(w_smem) + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = threadIdx.x >> 1, half = threadIdx.x & 1;
    const int64_t nkb = K / 128;
    const int64_t ntiles = (N / 128) * nkb;
    const int64_t step = gridDim.x;
    if (threadIdx.x == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        jet::ptx::fence_mbar_init();
    }
    __syncthreads();
    jet::griddep_launch_dependents();
    jet::griddep_wait();
    auto issue = [&](int st, int64_t t) {
        const int64_t nb = t / nkb, kb = t - nb * nkb;
        const uint32_t dst = base + st * kWTileBytes;
        mbar_arrive_expect_tx(&full[st], kWTileBytes);
        tma_load_2d(dst, &tmw, &full[st], (int32_t)(kb * 128), (int32_t)(nb * 128),
                    kStreamPolicy);
        tma_load_2d(dst + kWBoxBytes, &tmw, &full[st], (int32_t)(kb * 128 + 64),
                    (int32_t)(nb * 128), kStreamPolicy);
    };
    int64_t issued = 0;
    if (threadIdx.x == 0)
        for (int j = 0; j < 2 && blockIdx.x + j * step < ntiles; ++j, ++issued)
            issue(j, blockIdx.x + j * step);
    uint32_t it = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < ntiles; t += step, ++it) {
        const int st = it & 1;
        // A wait that gave up is agreed on at the barrier below, before any
        // global write; until then the (possibly incomplete) stage is only read.
        ok = mbar_wait(&full[st], (it >> 1) & 1u, nullptr, status, jet::SITE_QUANT_STAGE);
        const uint32_t box = base + st * kWTileBytes + half * kWBoxBytes;
        float f[64];  // -w; f[8k ..] holds chunk k ^ 4h of the row
#pragma unroll
        for (int k = 0; k < 8; ++k) unpack8_neg(lds128(swz128(box, row, k ^ (4 * half))), f + 8 * k);
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 64; i += 2) a = max_abs2(a, f[i], f[i + 1]);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
        if (lane == 0) warp_max[it & 1][warp] = a;
        if (__syncthreads_or(!ok)) {
            ok = false;
            break;
        }
        if (threadIdx.x == 0 && t + 2 * step < ntiles) {
            fence_proxy_async();
            issue(st, t + 2 * step);
            ++issued;
        }
        a = warp_max[it & 1][0];
#pragma unroll
        for (int i = 1; i < 8; ++i) a = fmaxf(a, warp_max[it & 1][i]);
        const float sc = group_scale(a);
        const Divisor d = make_divisor(sc);
        const int64_t nb = t / nkb, kb = t - nb * nkb;
        // f[16j ..] holds chunks 2(j ^ 2h) and 2(j ^ 2h) + 1: 16 bytes of codes
        uint4 *dst = reinterpret_cast<uint4 *>(q + (nb * 128 + row) * K + kb * 128 + half * 64);
        if (d.fast) {  // uniform over the block
#pragma unroll
            for (int j = 0; j < 4; ++j)
                dst[j ^ (2 * half)] =
                    make_uint4(encode4_fast(f + 16 * j, d), encode4_fast(f + 16 * j + 4, d),
                               encode4_fast(f + 16 * j + 8, d), encode4_fast(f + 16 * j + 12, d));
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                dst[j ^ (2 * half)] =
                    make_uint4(encode4(f + 16 * j, d), encode4(f + 16 * j + 4, d),
                               encode4(f + 16 * j + 8, d), encode4(f + 16 * j + 12, d));
        }
        if (threadIdx.x == 0) s[nb * nkb + kb] = sc;
    }
    if (!ok && threadIdx.x == 0)
        for (int64_t j = it; j < issued; ++j)
            mbar_wait(&full[j & 1], (uint32_t)(j >> 1) & 1u, nullptr, status,
                      jet::SITE_QUANT_STAGE);
    (void)N;
}

// ------------------------------------------------------------------ 128x1 --
// Persistent CTAs (two per SM, 256 threads) walk the (128 tokens x 128
// columns) tiles with a two-stage ring: each tile's 16 KB of codes arrive by
// one 2D TMA load and its 128 row scales by one bulk copy, both on the
// stage's mbarrier, and the load of the tile after next is issued as soon as
// the current tile has been read, so one tile is always in flight while
// another is computed.  Lane l of warp w owns columns 4l .. 4l+3 and tokens
// 16w .. 16w+15 (a warp reads one 128-byte token row per shared load, free
// of bank conflicts).  Pass 1 dequantizes -v = fl32(D4(q) * -s_row) (the
// negated product, exactly -v) into 64 registers and reduces the column
// maxima over its tokens; the 8 warps meet in shared memory, where 128
// threads turn the column maxima into the scales and their negated
// reciprocals (one column each).  Pass 2 divides the register-held values,
// converts, and writes each column's 16 codes as one 16-byte store into the
// transposed output.
constexpr int kRqThreads = 256;
constexpr int kRqCtasPerSm = 2;

// Pass 1 of a 128x1 tile: this thread's 4 columns x 16 tokens of a [128
// tokens][128 codes] shared-memory tile, dequantized and negated,
// -v = fl32(D4(q) * -s_row), into registers, and the column maxima over its
// tokens into col_max[w].  kSwz: the tile's 16-byte chunks are stored at
// chunk XOR (token % 8) (the fused quantizer writes it so; a TMA-loaded tile
// is plain).
template <bool kSwz>
__device__ __forceinline__ void rq_pass1(const uint32_t (*codes)[32], const float *srow,
                                         float (&v)[4][16], float (*col_max)[128], int lane,
                                         int w) {
    const int t0 = w * 16;
    float amax[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
        const float4 sr4 = *reinterpret_cast<const float4 *>(&srow[t0 + i]);
        const float sr[4] = {sr4.x, sr4.y, sr4.z, sr4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int t = t0 + i + u;
            const int word = kSwz ? ((((lane >> 2) ^ (t & 7)) << 2) | (lane & 3)) : lane;
            float d0, d1, d2, d3;
            e4m3x4_to_f32(codes[t][word], d0, d1, d2, d3);
            const float2 s2 = make_float2(-sr[u], -sr[u]);
            const float2 a = __fmul2_rn(make_float2(d0, d1), s2);
            const float2 b = __fmul2_rn(make_float2(d2, d3), s2);
            v[0][i + u] = a.x;
            v[1][i + u] = a.y;
            v[2][i + u] = b.x;
            v[3][i + u] = b.y;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            amax[j] = max_abs2(amax[j], v[j][i], v[j][i + 1]);
            amax[j] = max_abs2(amax[j], v[j][i + 2], v[j][i + 3]);
        }
    }
    *reinterpret_cast<float4 *>(&col_max[w][lane * 4]) =
        make_float4(amax[0], amax[1], amax[2], amax[3]);
}

// Between the passes, once col_max is complete: threads 0..127 turn the
// column maxima into the scales and negated reciprocals (one column each).
// Returns whether this thread's column takes the fast division (true for the
// other threads).
__device__ __forceinline__ bool rq_scales(const float (*col_max)[128], float *col_s,
                                          float *col_y) {
    if (threadIdx.x >= 128) return true;
    float a = col_max[0][threadIdx.x];
#pragma unroll
    for (int j = 1; j < 8; ++j) a = fmaxf(a, col_max[j][threadIdx.x]);
    const float sc = group_scale(a);
    const Divisor d = make_divisor(sc);
    col_s[threadIdx.x] = sc;
    col_y[threadIdx.x] = d.ny;
    return d.fast;
}

// Pass 2: quotients of the register-held values, each column's 16 codes as
// one 16-byte store into qT [K][M], the column scales into sT [M/128][K].
// `fast`: every column of the tile takes the fast division.
__device__ __forceinline__ void rq_pass2(const float (&v)[4][16], const float *col_s,
                                         const float *col_y, bool fast, int64_t M, int64_t K,
                                         int64_t mb, int64_t kb, uint8_t *__restrict__ qT,
                                         float *__restrict__ sT, int lane, int w) {
    const float4 s4 = *reinterpret_cast<const float4 *>(&col_s[lane * 4]);
    const float4 y4 = *reinterpret_cast<const float4 *>(&col_y[lane * 4]);
    const float scs[4] = {s4.x, s4.y, s4.z, s4.w};
    const float ys[4] = {y4.x, y4.y, y4.z, y4.w};
    const int64_t col = kb * 128 + lane * 4;
    uint8_t *dst = qT + col * M + mb * 128 + w * 16;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        Divisor d;
        d.s = scs[j];
        d.ny = ys[j];
        d.fast = scs[j] >= 0x1p-90f;
        uint32_t o[4];
        if (fast) {
#pragma unroll
            for (int g = 0; g < 4; ++g) o[g] = encode4_fast(&v[j][4 * g], d);
        } else {
#pragma unroll
            for (int g = 0; g < 4; ++g) o[g] = encode4(&v[j][4 * g], d);
        }
        *reinterpret_cast<uint4 *>(dst + (int64_t)j * M) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (w == 0) *reinterpret_cast<float4 *>(sT + mb * K + col) = s4;
}

__global__ void __launch_bounds__(kRqThreads, kRqCtasPerSm)
requant_128x1_kernel(const __grid_constant__ CUtensorMap tmq, const float *__restrict__ s,
                     int64_t M, int64_t K, uint8_t *__restrict__ qT,
                     float *__restrict__ sT, unsigned *status) {
    __shared__ __align__(128) uint32_t tile[2][128][32];  // [stage][token][4 codes]
    __shared__ __align__(16) float srow[2][128];
    __shared__ __align__(16) float col_max[8][128];
    __shared__ __align__(16) float col_s[128];
    __shared__ __align__(16) float col_y[128];
    __shared__ uint64_t full[2];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t nkb = K / 128;
    const int64_t ntiles = (M / 128) * nkb;
    const int64_t step = gridDim.x;
    if (threadIdx.x == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        jet::ptx::fence_mbar_init();
    }
    __syncthreads();
    jet::griddep_launch_dependents();
    jet::griddep_wait();
    // Tile t = mb * nkb + kb: CTAs running together take neighbouring column
    // blocks of the same 128 tokens.
    auto issue = [&](int st, int64_t t) {
        const int64_t mb = t / nkb, kb = t - mb * nkb;
        mbar_arrive_expect_tx(&full[st], 128u * 128u + 512u);
        tma_load_2d(smem_u32(&tile[st][0][0]), &tmq, &full[st], (int32_t)(kb * 128),
                    (int32_t)(mb * 128), kStreamPolicy);
        bulk_g2s(smem_u32(&srow[st][0]), s + kb * M + mb * 128, 512u, &full[st]);
    };
    int64_t issued = 0;  // loads issued (thread 0's count)
    if (threadIdx.x == 0)
        for (int j = 0; j < 2 && blockIdx.x + j * step < ntiles; ++j, ++issued)
            issue(j, blockIdx.x + j * step);
    uint32_t it = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < ntiles; t += step, ++it) {
        const int st = it & 1;
        // A wait that gave up is agreed on at the barrier below, before any
        // global write; until then the (possibly incomplete) stage is only read.
        ok = mbar_wait(&full[st], (it >> 1) & 1u, nullptr, status, jet::SITE_QUANT_STAGE);
        float v[4][16];
        rq_pass1<false>(tile[st], srow[st], v, col_max, lane, w);
        if (__syncthreads_or(!ok)) {
            ok = false;
            break;
        }
        // The stage has been read: refill it with the tile after next.
        if (threadIdx.x == 0 && t + 2 * step < ntiles) {
            jet::ptx::fence_proxy_async();
            issue(st, t + 2 * step);
            ++issued;
        }
        // Tiles whose every column takes the fast division (all but the
        // tiniest data) run pass 2 without a per-column test.
        const bool fast = __syncthreads_and(rq_scales(col_max, col_s, col_y));
        const int64_t mb = t / nkb, kb = t - mb * nkb;
        rq_pass2(v, col_s, col_y, fast, M, K, mb, kb, qT, sT, lane, w);
    }
    // After a time-out, loads still in flight must land before the CTA exits.
    if (!ok && threadIdx.x == 0)
        for (int64_t j = it; j < issued; ++j)
            mbar_wait(&full[j & 1], (uint32_t)(j >> 1) & 1u, nullptr, status,
                      jet::SITE_QUANT_STAGE);
}

// --------------------------------------------------- 1x128 and 128x1 fused --
// Both quantizations of one BF16 tensor (the output gradient) from a single
// read: per tile of 128 tokens x one K-block (two 64-column boxes with the
// 128-byte swizzle, 32 KB, two-stage TMA ring as above), phase A quantizes
// each token row as a 1x128 group (two threads per row, 64 values each, the
// row amax by one shuffle) and writes its codes and scale to global memory and
// to a shared-memory code tile (16-byte chunks at chunk XOR (row % 8): the
// stores are conflict-free per quarter-warp and the row reads of phase B still
// touch every bank once); phase B is the 128x1 re-quantization of that tile
// (rq_pass1/rq_scales/rq_pass2), i.e. from the FP8 values just written.  The
// results equal jet_quant_act_1x128 followed by jet_requant_128x1 bit for bit.
constexpr int kDualBoxBytes = 128 * 128;  // 128 rows x 64 BF16
constexpr int kDualTileBytes = 2 * kDualBoxBytes;
constexpr int kDualCtasPerSm = 2;
constexpr int kDualSmemBytes = 2 * kDualTileBytes + 1024;

__global__ void __launch_bounds__(256, kDualCtasPerSm)
quant_dual_kernel(const __grid_constant__ CUtensorMap tmx, int64_t M, int64_t K,
                  uint8_t *__restrict__ q, float *__restrict__ s, uint8_t *__restrict__ qT,
                  float *__restrict__ sT, unsigned *status) {
    extern __shared__ uint8_t dual_smem[];
    __shared__ __align__(128) uint32_t codes[128][32];
    __shared__ __align__(16) float srow[128];
    __shared__ __align__(16) float col_max[8][128];
    __shared__ __align__(16) float col_s[128];
    __shared__ __align__(16) float col_y[128];
    __shared__ uint64_t full[2];
    const uint32_t base = (smem_u32(dual_smem) + 1023u) & ~1023u;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int row = threadIdx.x >> 1, half = threadIdx.x & 1;
    const int64_t nkb = K / 128;
    const int64_t ntiles = (M / 128) * nkb;
    const int64_t step = gridDim.x;
    if (threadIdx.x == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        jet::ptx::fence_mbar_init();
    }
    __syncthreads();
    jet::griddep_launch_dependents();
    jet::griddep_wait();
    auto issue = [&](int st, int64_t t) {
        const int64_t mb = t / nkb, kb = t - mb * nkb;
        const uint32_t dst = base + st * kDualTileBytes;
        mbar_arrive_expect_tx(&full[st], kDualTileBytes);
        tma_load_2d(dst, &tmx, &full[st], (int32_t)(kb * 128), (int32_t)(mb * 128),
                    kStreamPolicy);
        tma_load_2d(dst + kDualBoxBytes, &tmx, &full[st], (int32_t)(kb * 128 + 64),
                    (int32_t)(mb * 128), kStreamPolicy);
    };
    int64_t issued = 0;
    if (threadIdx.x == 0)
        for (int j = 0; j < 2 && blockIdx.x + j * step < ntiles; ++j, ++issued)
            issue(j, blockIdx.x + j * step);
    uint32_t it = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < ntiles; t += step, ++it) {
        const int st = it & 1;
        ok = mbar_wait(&full[st], (it >> 1) & 1u, nullptr, status, jet::SITE_QUANT_STAGE);
        // phase A: the 1x128 group of token `row`, columns 64h .. 64h+63 here
        const uint32_t box = base + st * kDualTileBytes + half * kDualBoxBytes;
        float f[64];  // -x; f[8k ..] holds chunk k ^ 4h of the box row
#pragma unroll
        for (int k = 0; k < 8; ++k) unpack8_neg(lds128(swz128(box, row, k ^ (4 * half))), f + 8 * k);
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 64; i += 2) a = max_abs2(a, f[i], f[i + 1]);
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        if (__syncthreads_or(!ok)) {
            ok = false;
            break;
        }
        if (threadIdx.x == 0 && t + 2 * step < ntiles) {
            fence_proxy_async();
            issue(st, t + 2 * step);
            ++issued;
        }
        const int64_t mb = t / nkb, kb = t - mb * nkb;
        const int64_t m = mb * 128 + row;
        const float sc = group_scale(a);
        const Divisor d = make_divisor(sc);
        // f[16j ..] holds code chunk (16 codes) 4h + (j ^ 2h) of the row
        uint4 *gq = reinterpret_cast<uint4 *>(q + m * K + kb * 128 + half * 64);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint4 c;
            if (d.fast)
                c = make_uint4(encode4_fast(f + 16 * j, d), encode4_fast(f + 16 * j + 4, d),
                               encode4_fast(f + 16 * j + 8, d), encode4_fast(f + 16 * j + 12, d));
            else
                c = make_uint4(encode4(f + 16 * j, d), encode4(f + 16 * j + 4, d),
                               encode4(f + 16 * j + 8, d), encode4(f + 16 * j + 12, d));
            const int chunk = 4 * half + (j ^ (2 * half));
            gq[j ^ (2 * half)] = c;
            *reinterpret_cast<uint4 *>(&codes[row][(chunk ^ (row & 7)) * 4]) = c;
        }
        if (half == 0) {
            s[kb * M + m] = sc;
            srow[row] = sc;
        }
        __syncthreads();
        // phase B: 128x1 groups of the codes just written
        float v[4][16];
        rq_pass1<true>(codes, srow, v, col_max, lane, w);
        __syncthreads();
        const bool fast = __syncthreads_and(rq_scales(col_max, col_s, col_y));
        rq_pass2(v, col_s, col_y, fast, M, K, mb, kb, qT, sT, lane, w);
    }
    if (!ok && threadIdx.x == 0)
        for (int64_t j = it; j < issued; ++j)
            mbar_wait(&full[j & 1], (uint32_t)(j >> 1) & 1u, nullptr, status,
                      jet::SITE_QUANT_STAGE);
}

// Self-test of the division used above: q[i] = x[i] / s[i] through
// make_divisor + qdiv_neg, the same steps the quantizers take for a group
// scale.
__global__ void selftest_quotient_kernel(const float *__restrict__ x, const float *__restrict__ s,
                                         int64_t n, float *__restrict__ q) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        q[i] = qdiv_neg(-x[i], make_divisor(s[i]));
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// TMA coordinates are 32-bit: every tensor extent stays below 2^31.
constexpr int64_t kMaxRows = (int64_t)1 << 31;

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
// box_inner, zero fill outside (no swizzle unless asked).
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType type, uint32_t esize,
              uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * esize};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, type, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

jet_status jet_quant_act_1x128(const uint16_t *x, int64_t M, int64_t K, uint8_t *q,
                               float *s, jet_stream_t stream) {
    JET_REQUIRE(M >= 0 && K >= 0, JET_ERR_SHAPE);
    const bool empty = (M == 0 || K == 0);
    JET_REQUIRE(empty || (x && q && s), JET_ERR_NULL);
    JET_REQUIRE(K % 128 == 0 && M < kMaxRows && K < kMaxRows, JET_ERR_SHAPE);
    JET_REQUIRE(jet::aligned16(x) && jet::aligned16(q) && jet::aligned16(s), JET_ERR_ALIGN);
    jet::DeviceInfo dev;
    jet_status st = jet::current_device(&dev);
    if (st != JET_OK) return st;
    if (empty) return JET_OK;
    CUtensorMap tm;
    if (!make_map(&tm, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)K, (uint64_t)M, 64,
                  kActRowsPerCta, CU_TENSOR_MAP_SWIZZLE_128B))
        return JET_ERR_CUDA;
    const int64_t tiles = (M + kActRowsPerCta - 1) / kActRowsPerCta * (K / 128);
    const int64_t cap = (int64_t)dev.num_sms * kActCtasPerSm;
    return jet::launch_pdl(quant_act_1x128_kernel, dim3((unsigned)(tiles < cap ? tiles : cap)),
                           dim3(256), kActSmemBytes, jet::as_stream(stream), tm, M, K, q, s,
                           dev.status_word);
}

jet_status jet_quant_w_128x128(const uint16_t *w, int64_t N, int64_t K, uint8_t *q,
                               float *s, jet_stream_t stream) {
    JET_REQUIRE(N >= 0 && K >= 0, JET_ERR_SHAPE);
    const bool empty = (N == 0 || K == 0);
    JET_REQUIRE(empty || (w && q && s), JET_ERR_NULL);
    JET_REQUIRE(N % 128 == 0 && K % 128 == 0 && N < kMaxRows && K < kMaxRows, JET_ERR_SHAPE);
    JET_REQUIRE(jet::aligned16(w) && jet::aligned16(q) && jet::aligned16(s), JET_ERR_ALIGN);
    jet::DeviceInfo dev;
    jet_status st = jet::current_device(&dev);
    if (st != JET_OK) return st;
    if (empty) return JET_OK;
    static bool attr_set[64] = {};
    if (!attr_set[dev.ordinal]) {
        if (cudaFuncSetAttribute(quant_w_128x128_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kWSmemBytes) != cudaSuccess) {
            cudaGetLastError();
            return JET_ERR_CUDA;
        }
        attr_set[dev.ordinal] = true;
    }
    CUtensorMap tm;
    if (!make_map(&tm, w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)K, (uint64_t)N, 64, 128,
                  CU_TENSOR_MAP_SWIZZLE_128B))
        return JET_ERR_CUDA;
    const int64_t tiles = (N / 128) * (K / 128);
    const int64_t cap = (int64_t)dev.num_sms * kWCtasPerSm;
    return jet::launch_pdl(quant_w_128x128_kernel, dim3((unsigned)(tiles < cap ? tiles : cap)),
                           dim3(256), kWSmemBytes, jet::as_stream(stream), tm, N, K, q, s,
                           dev.status_word);
}

jet_status jet_requant_128x1(const uint8_t *q, const float *s, int64_t M, int64_t K,
                             uint8_t *qT, float *sT, jet_stream_t stream) {
    JET_REQUIRE(M >= 0 && K >= 0, JET_ERR_SHAPE);
    const bool empty = (M == 0 || K == 0);
    JET_REQUIRE(empty || (q && s && qT && sT), JET_ERR_NULL);
    JET_REQUIRE(M % 128 == 0 && K % 128 == 0 && M < kMaxRows && K < kMaxRows, JET_ERR_SHAPE);
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
    const int64_t tiles = (M / 128) * (K / 128);
    const int64_t cap = (int64_t)dev.num_sms * kRqCtasPerSm;
    return jet::launch_pdl(requant_128x1_kernel, dim3((unsigned)(tiles < cap ? tiles : cap)),
                           dim3(kRqThreads), 0, jet::as_stream(stream), tm, s, M, K, qT, sT,
                           dev.status_word);
}

jet_status jet_quant_dual_1x128_128x1(const uint16_t *x, int64_t M, int64_t K, uint8_t *q,
                                      float *s, uint8_t *qT, float *sT, jet_stream_t stream) {
    JET_REQUIRE(M >= 0 && K >= 0, JET_ERR_SHAPE);
    const bool empty = (M == 0 || K == 0);
    JET_REQUIRE(empty || (x && q && s && qT && sT), JET_ERR_NULL);
    JET_REQUIRE(M % 128 == 0 && K % 128 == 0 && M < kMaxRows && K < kMaxRows, JET_ERR_SHAPE);
    JET_REQUIRE(jet::aligned16(x) && jet::aligned16(q) && jet::aligned16(s) &&
                    jet::aligned16(qT) && jet::aligned16(sT),
                JET_ERR_ALIGN);
    jet::DeviceInfo dev;
    jet_status st = jet::current_device(&dev);
    if (st != JET_OK) return st;
    if (empty) return JET_OK;
    static bool attr_set[64] = {};
    if (!attr_set[dev.ordinal]) {
        if (cudaFuncSetAttribute(quant_dual_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kDualSmemBytes) != cudaSuccess) {
            cudaGetLastError();
            return JET_ERR_CUDA;
        }
        attr_set[dev.ordinal] = true;
    }
    CUtensorMap tm;
    if (!make_map(&tm, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)K, (uint64_t)M, 64, 128,
                  CU_TENSOR_MAP_SWIZZLE_128B))
        return JET_ERR_CUDA;
    const int64_t tiles = (M / 128) * (K / 128);
    const int64_t cap = (int64_t)dev.num_sms * kDualCtasPerSm;
    return jet::launch_pdl(quant_dual_kernel, dim3((unsigned)(tiles < cap ? tiles : cap)),
                           dim3(256), kDualSmemBytes, jet::as_stream(stream), tm, M, K, q, s, qT,
                           sT, dev.status_word);
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
