// Block-scaled FP8 GEMMs of the linear layer on the 5th-generation tensor
// core (tcgen05), one kernel template for the three products:
//
//   forward  Y [M][N] = sum_kb sx[kb][m]  * sw[n/128][kb]  * (qx  . qw^T)_kb
//   dgrad    dX[M][K] = sum_nb sdy[nb][m] * sw[nb][k/128]  * (qdy . qw)_nb
//   wgrad    dW[N][K] = sum_mb sdyT[mb][n] * sxT[mb][k]    * (qdyT . qxT^T)_mb
//
// ("Jet-RL ..." gist.science summary, "Quantisierungsschema": FP8 forward,
// DGrad and WGrad GEMMs; the scales are the FP32 per-group scales of the
// nmedialink page's quantization table.)  Because each 128-long slice of the
// contraction carries its own FP32 scales, the tensor core accumulates one
// slice at a time in TMEM and the epilogue warps fold it into FP32 registers
// with its row-scale x column-scale product.  MX block scaling (power-of-two
// scales per 32 elements) cannot represent these scales, so it is not used.
//
// Kernel organisation (persistent, one CTA per SM, 384 threads = 3 warpgroups):
//   warp 0     TMA producer: per 128-slice, one 128x128 A box and one 128xBN
//              B box (two 128x128 boxes for dgrad) into a ring of shared
//              memory stages with 128-byte swizzle, and the slice's FP32
//              scales (128 row scales, the column scales) into an 8-slot
//              ring by cp.async, so promotion never waits on global memory.
//   warp 1     allocates TMEM; warps 1 and 2 issue tcgen05.mma (K = 32 per
//              instruction, four per slice) into one of two TMEM accumulators
//              of BN columns (warp 1 the even slices, warp 2 the odd ones),
//              then commit to the stage's "empty" and the accumulator's
//              "full" barriers.
//   warp 3     pair kernel: issues each finished tile's TMA stores once the
//              promotion warps have staged it (a store's issue can hold its
//              thread for 800-1500 cycles); otherwise idle.
//              Warpgroup 0 (warps 0-3) gives registers back
//              (setmaxnreg 72) so that the epilogue warpgroups can hold their
//              accumulators and three TMEM load buffers (setmaxnreg 216;
//              200 and two buffers for the grouped products):
//              128*72 + 256*216 = 384 * 168, the allocation the block is
//              launched with.
//   warps 4-11 promotion/epilogue: two warpgroups split the tile's columns;
//              each thread owns one output row (its TMEM lane) and BN/2 FP32
//              accumulators, loads each slice from TMEM, applies the scales,
//              releases the accumulator, and after the last slice writes
//              BF16 (round to nearest even).
// Operand majorness: A is always K-major (contraction contiguous).  B is
// K-major for forward and wgrad; for dgrad the weight codes qw[N][K] are read
// as they are, MN-major (the output column contiguous), so no transposed copy
// of the weights is needed.
// Split contraction (at most 512 output rows, as in rollout decode): such a
// problem has only a few C/BN-wide tiles, far fewer than the 152 SMs, so the
// contraction is cut into `splits` contiguous ranges of 128-slices, one work
// unit per (tile, range).  Each unit writes its FP32
// partial tile to a caller-provided workspace [splits][R][C]; a second kernel
// adds the partials in split order (deterministic) and rounds once to BF16.
// Every mbarrier wait is bounded by kWaitLimitCycles SM cycles (~2 s at the
// maximum clock; jet_common.cuh), except the pipeline waits of the time-out
// self-test (kFwdTimeoutTest), which poll against a limit given at launch.  A
// role that gives up records JET_ERR_TIMEOUT and sets the CTA's abort flag;
// the CTA's other roles stop at their next wait, in-flight copies and MMAs are
// drained and TMEM is freed before the kernel returns.  The abort flag is per
// CTA: in a CTA pair the peer learns of it only through its own waits running
// out.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "jet_common.cuh"
#include "sm100_ptx.cuh"

namespace {

using namespace jet;
using namespace jet::ptx;

// The grouped modes run the product of several expert linears in one launch
// (tokens concatenated in expert order, weights stacked [E][N][K]):
// kFwdGrouped and kDgradGrouped split the rows by expert, kWgradGrouped the
// contraction (each expert's dW over its own tokens, outputs stacked).
// kFwdTimeoutTest is the forward product of the time-out self-test: its
// pipeline waits poll (mbar_wait_polled) against a limit given at launch.
enum Mode {
    kFwd = 0, kDgrad = 1, kWgrad = 2, kFwdGrouped = 3, kDgradGrouped = 4, kWgradGrouped = 5,
    kFwdTimeoutTest = 6
};
constexpr int base_mode(int mode) {
    return mode == kFwdGrouped || mode == kFwdTimeoutTest ? kFwd
           : mode == kDgradGrouped                        ? kDgrad
           : mode == kWgradGrouped                        ? kWgrad
                                                          : mode;
}
constexpr bool is_grouped(int mode) {
    return mode == kFwdGrouped || mode == kDgradGrouped || mode == kWgradGrouped;
}
constexpr int kMaxGroups = 384;  // one expert per thread of the unit-count scan

constexpr int kThreads = 384;
static_assert(kMaxGroups <= kThreads, "the unit-count scan takes one expert per thread");
constexpr uint32_t kRegsControl = 72;    // warpgroup 0 after setmaxnreg
constexpr uint32_t kRegsEpilogue = 216;  // warpgroups 1-2 after setmaxnreg
// the grouped products, whose expert tables already take registers, keep
// 200 and two TMEM load buffers: at 216 their kernels spilled
constexpr uint32_t kRegsEpilogueGrouped = 200;
static_assert(128 * kRegsControl + 256 * kRegsEpilogue <= kThreads * 168 &&
                  128 * kRegsControl + 256 * kRegsEpilogueGrouped <= kThreads * 168,
              "register split exceeds the launch allocation");
constexpr int BM = 128;  // output rows per tile (TMEM lanes)
constexpr int BK = 128;  // contraction slice = one scale block

template <int BN, int CL, bool STAGED, int ST = 0>
struct Cfg {
    // Per CTA and stage: A's 128 rows and B's BN (CL = 1) or BN/2 (pair) rows.
    static constexpr int kBRows = BN / CL;
    static constexpr int kABytes = BM * BK;
    static constexpr int kBBytes = kBRows * BK;
    static constexpr int kStageBytes = kABytes + kBBytes;
    // Scale ring: per slice, the tile's 128 row scales and its column scales
    // (BN per-column values for wgrad, BN/128 block values otherwise).
    static constexpr int kScaleSlots = 8;
    static constexpr int kScaleRowBytes = BM * 4;
    static constexpr int kScaleSlotBytes = kScaleRowBytes + BN * 4;
    // Output staging (STAGED: the pair kernel and the grouped forward): each
    // promotion warp's 32 x 128 BF16 block, 128-byte swizzled, written out by
    // TMA stores, so that the promotion warps go back to the accumulators
    // while the stores drain.
    static constexpr int kOutWarpBytes = 32 * 128 * 2;
    static constexpr int kOutBytes = STAGED ? 8 * kOutWarpBytes : 0;
    // four operand stages where they fit beside the staging, else three;
    // ST > 0 asks for ST stages (the deep split-contraction kernel: six
    // 32 KB stages keep 96 KB of weights in flight per SM)
    static constexpr int kStages =
        ST > 0 ? ST
               : (4 * kStageBytes + kOutBytes + kScaleSlots * kScaleSlotBytes + 1024 <= 227 * 1024
                      ? 4
                      : 3);
    static constexpr int kSmemBytes = kStages * kStageBytes + kOutBytes +
                                      kScaleSlots * kScaleSlotBytes + 1024;  // + alignment slack
    static constexpr int kTmemCols = 2 * BN;                           // two accumulators
    static constexpr int kHalf = BN / 2;  // columns per epilogue thread
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// Tile order: 0 = column tiles fastest (B stays in L2, A read once),
// 1 = row tiles fastest (A stays in L2, B read once), 2 = groups of `g` row
// tiles, row tiles fastest inside a group (the group's A stays in L2, B is
// read once per group), 3 = groups of `g` column tiles, column tiles fastest
// inside a group (the group's B stays in L2, A is read once per group).
struct Raster {
    int mode;
    int g;
};

__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, Raster r, int &mt,
                                            int &nt) {
    if (r.mode == 0) {
        mt = t / tiles_n;
        nt = t - mt * tiles_n;
    } else if (r.mode == 1) {
        nt = t / tiles_m;
        mt = t - nt * tiles_m;
    } else if (r.mode == 2) {
        const int per_group = r.g * tiles_n;
        const int g = t / per_group;
        const int within = t - g * per_group;
        const int rows = min(r.g, tiles_m - g * r.g);
        nt = within / rows;
        mt = g * r.g + (within - nt * rows);
    } else {
        const int per_group = r.g * tiles_m;
        const int g = t / per_group;
        const int within = t - g * per_group;
        const int cols = min(r.g, tiles_n - g * r.g);
        mt = within / cols;
        nt = g * r.g + (within - mt * cols);
    }
}

// Work unit t -> its tile and its range [kb0, kb1) of 128-slices.  The
// `splits` ranges of one tile are consecutive units; each range is non-empty
// because splits <= nkb.
__device__ __forceinline__ void unit_coords(int t, int splits, int nkb, int tiles_m, int tiles_n,
                                            Raster r, int &mt, int &nt, int &kb0, int &kb1) {
    if (splits == 1) {  // the common case, without its two divisions
        tile_coords(t, tiles_m, tiles_n, r, mt, nt);
        kb0 = 0;
        kb1 = nkb;
        return;
    }
    const int tile = t / splits, sp = t - tile * splits;
    tile_coords(tile, tiles_m, tiles_n, r, mt, nt);
    kb0 = sp * nkb / splits;
    kb1 = (sp + 1) * nkb / splits;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// acc[base .. base+7] += p[2j .. 2j+1] * sc  (pairs, fma.rn.f32x2)
template <int N>
__device__ __forceinline__ void promote16(float2 (&acc)[N], int base, const uint32_t (&p)[16],
                                          float2 sc) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
        acc[base + j] = __ffma2_rn(
            make_float2(__uint_as_float(p[2 * j]), __uint_as_float(p[2 * j + 1])), sc,
            acc[base + j]);
}

// acc[base .. base+7] += (p * rs) * cs   (per-column scales, wgrad; cs holds
// this chunk's 16 column scales)
template <int N>
__device__ __forceinline__ void promote16_cols(float2 (&acc)[N], int base,
                                               const uint32_t (&p)[16], float2 rs,
                                               const float4 (&cs)[4]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 t0 = __fmul2_rn(
            make_float2(__uint_as_float(p[4 * q + 0]), __uint_as_float(p[4 * q + 1])), rs);
        const float2 t1 = __fmul2_rn(
            make_float2(__uint_as_float(p[4 * q + 2]), __uint_as_float(p[4 * q + 3])), rs);
        acc[base + 2 * q] = __ffma2_rn(t0, make_float2(cs[q].x, cs[q].y), acc[base + 2 * q]);
        acc[base + 2 * q + 1] =
            __ffma2_rn(t1, make_float2(cs[q].z, cs[q].w), acc[base + 2 * q + 1]);
    }
}

__device__ __forceinline__ void load_cs(float4 (&cs)[4], const float *src) {
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) cs[q] = s4[q];
}

// CL = 1: one CTA computes a 128 x BN tile with tcgen05.mma.cta_group::1.
// CL = 2: a cluster of two CTAs computes a 256 x BN tile with the pair MMA
// (tcgen05.mma.cta_group::2) issued by the even CTA ("leader"): each CTA loads
// its own 128 rows of A and half of B's BN rows, so each SM takes in 32 KB per
// 128-slice instead of 48 KB and six stages fit in shared memory instead of
// four.  Both CTAs' TMA loads signal the leader's "full" barrier; the
// leader's commits arrive on both CTAs' "empty" and "TMEM full" barriers; both
// CTAs' promotion warps release the leader's "TMEM empty" barrier; each CTA
// promotes and stores its own 128 rows from its own TMEM.
template <int BN, int MODE, int CL, int ST = 0>
__global__ void __launch_bounds__(kThreads, 1)
gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmY, const float *__restrict__ sa,
                const float *__restrict__ sb,
                uint16_t *__restrict__ out, int R, int C, int D, Raster raster, int splits,
                float *__restrict__ partial, const int64_t *__restrict__ goff, int gE,
                unsigned *status, uint64_t wait_limit) {
    using CF = Cfg<BN, CL, CL == 2 || is_grouped(MODE), ST>;
    constexpr int S = CF::kStages;
    // MMA-issuing warps (see the MMA role): two when every stage and every
    // TMEM accumulator is used by one issuer only, i.e. an even stage count.
    constexpr uint32_t kIssuers = S % 2 == 0 ? 2u : 1u;
    constexpr int SS = CF::kScaleSlots;
    constexpr bool kPair = CL == 2;
    constexpr uint16_t kPairMask = 0x3;
    extern __shared__ uint8_t dyn_smem[];
    __shared__ uint64_t full_bar[S], empty_bar[S], tfull_bar[2], tempty_bar[2], drain_bar;
    // Output stores of the pair kernel: the promotion warps stage a tile and
    // arrive on "staged"; warp 3 issues the TMA stores, waits until they have
    // read the staging buffers and arrives on "staging free".
    constexpr bool kStoreWarp = CL == 2 && !is_grouped(MODE);
    __shared__ uint64_t staged_bar, sfree_bar;
    __shared__ uint64_t sfull_bar[SS], sempty_bar[SS];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    // grouped forward: per expert, its first row and the prefix of its units
    constexpr bool kGrp = is_grouped(MODE);
    constexpr int BASE = base_mode(MODE);
    constexpr bool kFwdLike = BASE == kFwd;
    constexpr int kGT = kGrp ? kMaxGroups + 1 : 1;
    __shared__ int g_off[kGT], g_pre[kGT];
    __shared__ int g_warp[kThreads / 32];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t smem_base = (smem_u32(dyn_smem) + 1023u) & ~1023u;
    const uint32_t out_base = smem_base + S * CF::kStageBytes;  // 1024-aligned
    const uint32_t scale_base = out_base + CF::kOutBytes;
    const int tiles_m = (R + BM - 1) / BM;
    const int tiles_n = C / BN;
    const int units_m = (tiles_m + CL - 1) / CL;  // row tiles per cluster step
    int total = units_m * tiles_n * splits;  // work units: (tile, contraction range)
    const int nkb = D / BK;
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int unit0 = blockIdx.x / CL, unit_step = gridDim.x / CL;
    volatile int *abort = &abort_sh;
    // Pipeline waits (abortable): bounded by kWaitLimitCycles, or by the
    // launch's `wait_limit` with polling in the time-out self-test.
    auto pwait = [&](uint64_t *bar, uint32_t parity, unsigned site) -> bool {
        if constexpr (MODE == kFwdTimeoutTest)
            return mbar_wait_polled(bar, parity, abort, status, site, wait_limit);
        else
            return mbar_wait(bar, parity, abort, status, site);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int s = 0; s < SS; ++s) {
            mbar_init(&sfull_bar[s], 32);  // one cp.async arrival per producer lane
            mbar_init(&sempty_bar[s], 8);  // one arrival per epilogue warp
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull_bar[b], 1);
            mbar_init(&tempty_bar[b], 8 * CL);  // epilogue warps of every CTA of the pair
        }
        mbar_init(&drain_bar, kIssuers);  // one drain commit per MMA-issuing warp
        mbar_init(&staged_bar, 8);         // one arrival per epilogue warp
        mbar_init(&sfree_bar, 1);          // the store warp
        abort_sh = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        if (kPair) {
            tmem_alloc_pair(&tmem_base_sh, CF::kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&tmem_base_sh, CF::kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    if (kPair)
        cluster_sync();  // the peer's barriers are initialised before any remote use
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    griddep_launch_dependents();
    griddep_wait();
    if (kGrp) {
        // Expert e owns tokens off[e] .. off[e+1], clamped to the token
        // count (R, or D for WGrad) so that nothing outside the operands
        // and the output is ever touched.  Forward / DGrad: the expert's
        // rows make ceil(rows / 128) * tiles_n units; one expert per thread,
        // then a block-wide inclusive scan of the unit counts.  WGrad: every
        // expert has the same units (its whole dW).
        const int i = threadIdx.x;
        const int glim = BASE == kWgrad ? D : R;
        auto clampr = [&](int64_t v) { return (int)(v < 0 ? 0 : (v > glim ? glim : v)); };
        int cnt = 0;
        for (int j = i; j <= gE; j += kThreads) g_off[j] = clampr(goff[j]);  // gE + 1 entries
        if (BASE != kWgrad && i < gE) {
            const int rows = clampr(goff[i + 1]) - clampr(goff[i]);
            cnt = rows > 0 ? (rows + BM - 1) / BM * tiles_n : 0;
        }
        int incl = cnt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        if (lane == 31) g_warp[warp] = incl;
        __syncthreads();
        int before = 0;
        for (int j = 0; j < warp; ++j) before += g_warp[j];
        if (i < gE) g_pre[i + 1] = before + incl;
        if (i == 0) g_pre[0] = 0;
        __syncthreads();
        total = BASE == kWgrad ? gE * units_m * tiles_n : g_pre[gE];
    }
    // Work unit t -> row tile origin m0 (row of A), column origin n0, its
    // slice range, the expert whose weights it uses, and in output rows its
    // origin mo and row limit rlim.
    auto coords = [&](int t, int &m0, int &n0, int &kb0, int &kb1, int &grp, int &mo,
                      int &rlim) {
        if (kGrp && BASE == kWgrad) {
            const int per = units_m * tiles_n;
            grp = t / per;
            const int u = t - grp * per, mu = u / tiles_n;
            m0 = (mu * CL + (int)rank) * BM;
            n0 = (u - mu * tiles_n) * BN;
            kb0 = g_off[grp] / BK;
            kb1 = (g_off[grp + 1] > g_off[grp] ? g_off[grp + 1] : g_off[grp]) / BK;
            mo = grp * R + m0;
            rlim = grp * R + R;
        } else if (kGrp) {
            int lo = 0, hi = gE - 1;  // the expert e with g_pre[e] <= t < g_pre[e+1]
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (g_pre[mid] <= t) lo = mid; else hi = mid - 1;
            }
            const int u = t - g_pre[lo], mt = u / tiles_n;
            grp = lo;
            m0 = g_off[lo] + mt * BM;
            n0 = (u - mt * tiles_n) * BN;
            rlim = g_off[lo + 1] > g_off[lo] ? g_off[lo + 1] : g_off[lo];
            kb0 = 0;
            kb1 = nkb;
            mo = m0;
        } else {
            int mu, nt;
            unit_coords(t, splits, nkb, units_m, tiles_n, raster, mu, nt, kb0, kb1);
            m0 = (mu * CL + (int)rank) * BM;
            n0 = nt * BN;
            rlim = R;
            grp = 0;
            mo = m0;
        }
    };

    // Each role is nested inside its own setmaxnreg branch so that the
    // register limit of one branch never applies to the other.
    if (warp < 4) {
        reg_dealloc<kRegsControl>();
        if (warp == 0) {
            // -------------------------------------------------- TMA producer
            // The operand that the tile order walks again (modes 0, 3: B;
            // modes 1, 2: A) is kept in L2; the other streams.
            const uint64_t keep = policy_evict_last(), stream_once = policy_evict_first();
            const bool keep_b = raster.mode == 0 || raster.mode == 3;
            const uint64_t pol_a = keep_b ? stream_once : keep;
            const uint64_t pol_b = keep_b ? keep : stream_once;
            uint32_t it = 0;
            bool ok = true;
            for (int t = unit0; ok && t < total; t += unit_step) {
                int m0, n0, kb0, kb1, grp, mo, rlim;
                coords(t, m0, n0, kb0, kb1, grp, mo, rlim);
                // the expert's weights in the stacked B: rows (forward) or,
                // read MN-major, the contraction axis (DGrad)
                const int brow0 = kGrp && BASE == kFwd ? grp * C : 0;
                const int bk0 = kGrp && BASE == kDgrad ? grp * D : 0;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % S;
                    const uint32_t use = it / S;
                    const int ss = it % SS;
                    const uint32_t suse = it / SS;
                    if (!pwait(&empty_bar[s], (use & 1u) ^ 1u, SITE_GEMM_PRODUCER_EMPTY) ||
                        !pwait(&sempty_bar[ss], (suse & 1u) ^ 1u, SITE_GEMM_PRODUCER_EMPTY)) {
                        ok = false;
                        break;
                    }
                    // Scales of this slice -> scale slot ss (all 32 lanes).
                    const uint32_t slot = scale_base + ss * CF::kScaleSlotBytes;
                    const float *srow = sa + (size_t)kb * R;
#pragma unroll
                    for (int j = 0; j < BM / 32; ++j) {
                        const int r = m0 + lane + 32 * j;
                        cp_async4(slot + (lane + 32 * j) * 4, srow + (r < R ? r : R - 1),
                                  r < R ? 4u : 0u);
                    }
                    const uint32_t scol = slot + CF::kScaleRowBytes;
                    if (BASE == kWgrad) {
                        const float *src = sb + (size_t)kb * C + n0;
#pragma unroll
                        for (int j = 0; j < BN / 128; ++j)
                            cp_async16(scol + (lane + 32 * j) * 16, src + 4 * (lane + 32 * j));
                    } else if (lane < BN / 128) {
                        const float *src =
                            kFwdLike ? sb + ((size_t)grp * (C / 128) + n0 / 128 + lane) * nkb + kb
                                     : sb + ((size_t)grp * nkb + kb) * (C / 128) + n0 / 128 + lane;
                        cp_async4(scol + lane * 4, src, 4u);
                    }
                    cp_async_arrive_noinc(&sfull_bar[ss]);
                    if (lane == 0) {
                        const uint32_t a_s = smem_base + s * CF::kStageBytes;
                        const uint32_t b_s = a_s + CF::kABytes;
                        if (kPair) {
                            // Both CTAs' boxes complete on the leader's barrier,
                            // which expects the pair's bytes.
                            const uint32_t fb = map_to_cta(&full_bar[s], 0);
                            if (leader) mbar_arrive_expect_tx(&full_bar[s], 2 * CF::kStageBytes);
                            tma_load_2d_pair(a_s, &tmA, fb, kb * BK, m0, pol_a);
                            if (BASE == kDgrad)
                                tma_load_2d_pair(b_s, &tmB, fb, n0 + CF::kBRows * (int)rank,
                                                 bk0 + kb * BK, pol_b);
                            else
                                tma_load_2d_pair(b_s, &tmB, fb, kb * BK,
                                                 brow0 + n0 + CF::kBRows * (int)rank, pol_b);
                        } else {
                            mbar_arrive_expect_tx(&full_bar[s], CF::kStageBytes);
                            tma_load_2d(a_s, &tmA, &full_bar[s], kb * BK, m0, pol_a);
                            if (BASE == kDgrad) {
#pragma unroll
                                for (int h = 0; h < BN / 128; ++h)
                                    tma_load_2d(b_s + h * 128 * BK, &tmB, &full_bar[s],
                                                n0 + 128 * h, bk0 + kb * BK, pol_b);
                            } else {
                                tma_load_2d(b_s, &tmB, &full_bar[s], kb * BK, brow0 + n0,
                                            pol_b);
                            }
                        }
                    }
                    __syncwarp();
                }
            }
            // Every issued load must have landed before the CTA can exit (the
            // pair's loads are tracked by the leader's barriers).
            if (!kPair || leader)
                for (uint32_t j = it > (uint32_t)S ? it - S : 0u; j < it; ++j)
                    mbar_wait(&full_bar[j % S], (j / S) & 1u, nullptr, status, SITE_GEMM_DRAIN);
            for (uint32_t j = it > (uint32_t)SS ? it - SS : 0u; j < it; ++j)
                mbar_wait(&sfull_bar[j % SS], (j / SS) & 1u, nullptr, status, SITE_GEMM_DRAIN);
        } else if ((warp == 1 || (warp == 2 && kIssuers == 2)) && leader) {
            // -------------------------------------------------- MMA issuers
            // (in a pair only the leader issues; the MMA spans both CTAs)
            // Warp 1 issues the even slices (TMEM accumulator 0), warp 2 the
            // odd ones (accumulator 1).  A thread that issues tcgen05.mma while
            // the tensor core's queue is full stalls there, about 128 cycles
            // per MMA, and holds back the other warps of its SM sub-partition
            // (here promotion warps, the critical path); two issuers halve that
            // per sub-partition.  Each warp's slices use one accumulator and
            // (S even) every second stage, so each warp waits on each
            // barrier's phases in order; with an odd stage count, or a third
            // issuer, a warp would skip a phase, whose parity then aliases the
            // one before, so those configurations keep a single issuer.
            const uint32_t mw = (uint32_t)(warp - 1);
            constexpr bool kMN = BASE == kDgrad;
            constexpr uint32_t kIdesc =
                kPair ? idesc_e4m3_f32(2 * BM, BN, kMN) : idesc_e4m3_f32(BM, kMN ? 128 : BN, kMN);
            uint32_t it = 0;
            bool ok = true;
            for (int t = unit0; ok && t < total; t += unit_step) {
                int m0, n0, kb0, kb1, grp, mo, rlim;
                coords(t, m0, n0, kb0, kb1, grp, mo, rlim);
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    if (it % kIssuers != mw) continue;  // the other issuer's slice
                    const int s = it % S;
                    const uint32_t use = it / S;
                    const int buf = it & 1;
                    const uint32_t tuse = it >> 1;
                    if (!pwait(&tempty_bar[buf], (tuse & 1u) ^ 1u, SITE_GEMM_MMA_TMEM_EMPTY) ||
                        !pwait(&full_bar[s], use & 1u, SITE_GEMM_MMA_FULL)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint32_t a_s = smem_base + s * CF::kStageBytes;
                        const uint32_t b_s = a_s + CF::kABytes;
                        const uint32_t d = tmem + buf * BN;
#pragma unroll
                        for (int ks = 0; ks < BK / 32; ++ks) {
                            const uint64_t adesc = smem_desc(a_s + ks * 32, 16, 1024, kSwizzle128B);
                            if (kPair) {
                                // per CTA: B holds BN/2 rows (K-major) or one
                                // 128-column MN-major atom (dgrad)
                                const uint64_t bdesc =
                                    kMN ? smem_desc(b_s + ks * 32 * 128, 1024, 1024, kSwizzle128B)
                                        : smem_desc(b_s + ks * 32, 16, 1024, kSwizzle128B);
                                mma_e4m3_pair(d, adesc, bdesc, kIdesc, ks > 0);
                            } else if (kMN) {
                                // MN-major B: 8-row contraction groups 1024 B apart;
                                // each MMA covers one 128-column swizzle atom.
#pragma unroll
                                for (int h = 0; h < BN / 128; ++h) {
                                    const uint64_t bdesc =
                                        smem_desc(b_s + h * 128 * BK + ks * 32 * 128, 1024, 1024,
                                                  kSwizzle128B);
                                    mma_e4m3(d + h * 128, adesc, bdesc, kIdesc, ks > 0);
                                }
                            } else {
                                const uint64_t bdesc =
                                    smem_desc(b_s + ks * 32, 16, 1024, kSwizzle128B);
                                mma_e4m3(d, adesc, bdesc, kIdesc, ks > 0);
                            }
                        }
                        if (kPair) {
                            mma_commit_pair_mc(&empty_bar[s], kPairMask);
                            mma_commit_pair_mc(&tfull_bar[buf], kPairMask);
                        } else {
                            mma_commit(&empty_bar[s]);
                            mma_commit(&tfull_bar[buf]);
                        }
                    }
                    __syncwarp();
                }
            }
            // All issued MMAs must complete before TMEM is released.
            if (lane == 0) {
                if (kPair)
                    mma_commit_pair_mc(&drain_bar, 0x1);
                else
                    mma_commit(&drain_bar);
            }
            __syncwarp();
            mbar_wait(&drain_bar, 0, nullptr, status, SITE_GEMM_DRAIN);
        } else if (warp == 3 && kStoreWarp) {
            // -------------------------------------------------- output stores
            // Issuing a TMA store can hold the issuing thread for 800-1500
            // cycles (measured) while the TMA unit works through the operand
            // loads; here that wait is off the promotion warps' path.
            uint32_t j = 0;
            for (int t = unit0; t < total; t += unit_step, ++j) {
                int m0, n0, kb0, kb1, grp, mo, rlim;
                coords(t, m0, n0, kb0, kb1, grp, mo, rlim);
                if (!pwait(&staged_bar, j & 1u, SITE_GEMM_EPI_TMEM_FULL)) break;
                if (lane == 0) {
                    const uint64_t pol_out = policy_evict_first();  // not re-read here
#pragma unroll 1
                    for (int ew = 0; ew < 8; ++ew) {
                        const uint32_t wbuf = out_base + ew * CF::kOutWarpBytes;
                        const int col0 = n0 + (ew >> 2) * CF::kHalf, row0 = mo + (ew & 3) * 32;
#pragma unroll
                        for (int h = 0; h < CF::kHalf / 64; ++h)
                            tma_store_2d_hint(&tmY, wbuf + 4096 * h, col0 + 64 * h, row0, pol_out);
                    }
                    bulk_commit_group();
                    bulk_wait_group_read0();  // the staging buffers have been read
                    mbar_arrive(&sfree_bar);
                }
                __syncwarp();
            }
            if (lane == 0) bulk_wait_group0();  // every store complete before exit
        }
    } else {
        reg_alloc<kGrp ? kRegsEpilogueGrouped : kRegsEpilogue>();
        // ----------------------------------------- promotion and epilogue
        constexpr int H = CF::kHalf;
        constexpr int NCH = H / 16;
        const int ew = warp - 4;
        const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
        const int ch = ew >> 2;     // column half
        const uint64_t pol_out = policy_evict_first();  // outputs are not re-read here
        uint32_t tempty_remote[2] = {0u, 0u};
        if (kPair) {
            tempty_remote[0] = map_to_cta(&tempty_bar[0], 0);
            tempty_remote[1] = map_to_cta(&tempty_bar[1], 0);
        }
        uint32_t it = 0;
        bool ok = true;
        uint32_t tile_j = 0;  // this CTA's tiles so far (store-warp hand-off phases)
        for (int t = unit0; ok && t < total; t += unit_step, ++tile_j) {
            int m0, n0, kb0, kb1, grp, mo, rlim;
            coords(t, m0, n0, kb0, kb1, grp, mo, rlim);
            const int row = mo + quad * 32 + lane;  // output row
            const bool row_ok = row < rlim;
            const int col0 = n0 + ch * H;
            float2 acc[H / 2];
#pragma unroll
            for (int i = 0; i < H / 2; ++i) acc[i] = make_float2(0.0f, 0.0f);

            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int buf = it & 1;
                const uint32_t tuse = it >> 1;
                const int ss = it % SS;
                const uint32_t suse = it / SS;
                if (!pwait(&sfull_bar[ss], suse & 1u, SITE_GEMM_EPI_TMEM_FULL)) {
                    ok = false;
                    break;
                }
                const float *slot = reinterpret_cast<const float *>(
                    dyn_smem + (scale_base - smem_u32(dyn_smem)) + ss * CF::kScaleSlotBytes);
                const float rs = slot[quad * 32 + lane];
                const float *scol = slot + BM;
                float sc = 0.0f;
                if (BASE != kWgrad) {
                    sc = rs * scol[(ch * H) / 128];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sempty_bar[ss]);
                }
                if (!pwait(&tfull_bar[buf], tuse & 1u, SITE_GEMM_EPI_TMEM_FULL)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + buf * BN + ch * H;
                if constexpr (!kGrp) {
                    // Three 16-column buffers: a wait (which covers every TMEM
                    // load of the thread) comes every second chunk, after two
                    // chunks of arithmetic, instead of after each one.
                    uint32_t pb[3][16];
                    tmem_ld16(taddr, pb[0]);
                    if (NCH > 1) tmem_ld16(taddr + 16, pb[1]);
                    tmem_ld_wait(pb[0]);
                    if (NCH > 1) tmem_ld_pin(pb[1]);
                    if (BASE != kWgrad) {
                        const float2 sc2 = make_float2(sc, sc);
    #pragma unroll
                        for (int c = 0; c < NCH; c += 2) {
                            if (c + 2 < NCH) tmem_ld16(taddr + (c + 2) * 16, pb[(c + 2) % 3]);
                            promote16(acc, c * 8, pb[c % 3], sc2);
                            if (c + 3 < NCH) tmem_ld16(taddr + (c + 3) * 16, pb[c % 3]);
                            promote16(acc, (c + 1) * 8, pb[(c + 1) % 3], sc2);
                            if (c + 2 < NCH) {
                                tmem_ld_wait(pb[(c + 2) % 3]);
                                if (c + 3 < NCH) tmem_ld_pin(pb[c % 3]);
                            }
                        }
                    } else {
                        // Column scales are loaded one chunk ahead of their use so
                        // that shared-memory latency overlaps the previous chunk.
                        const float *cs = scol + ch * H;
                        const float2 rs2 = make_float2(rs, rs);
                        float4 csa[4], csb[4];
                        load_cs(csa, cs);
    #pragma unroll
                        for (int c = 0; c < NCH; c += 2) {
                            if (c + 2 < NCH) tmem_ld16(taddr + (c + 2) * 16, pb[(c + 2) % 3]);
                            load_cs(csb, cs + (c + 1) * 16);
                            promote16_cols(acc, c * 8, pb[c % 3], rs2, csa);
                            if (c + 3 < NCH) tmem_ld16(taddr + (c + 3) * 16, pb[c % 3]);
                            if (c + 2 < NCH) load_cs(csa, cs + (c + 2) * 16);
                            promote16_cols(acc, (c + 1) * 8, pb[(c + 1) % 3], rs2, csb);
                            if (c + 2 < NCH) {
                                tmem_ld_wait(pb[(c + 2) % 3]);
                                if (c + 3 < NCH) tmem_ld_pin(pb[c % 3]);
                            }
                        }
                    }
                } else {
                    // The grouped products keep two buffers and a wait per
                    // chunk (their register budget has no room for a third).
                    uint32_t p0[16], p1[16];
                    tmem_ld16(taddr, p0);
                    if (BASE != kWgrad) {
                        const float2 sc2 = make_float2(sc, sc);
#pragma unroll
                        for (int c = 0; c < NCH; c += 2) {
                            tmem_ld_wait(p0);
                            tmem_ld16(taddr + (c + 1) * 16, p1);
                            promote16(acc, c * 8, p0, sc2);
                            tmem_ld_wait(p1);
                            if (c + 2 < NCH) tmem_ld16(taddr + (c + 2) * 16, p0);
                            promote16(acc, (c + 1) * 8, p1, sc2);
                        }
                    } else {
                        const float *cs = scol + ch * H;
                        const float2 rs2 = make_float2(rs, rs);
                        float4 csa[4], csb[4];
                        load_cs(csa, cs);
#pragma unroll
                        for (int c = 0; c < NCH; c += 2) {
                            load_cs(csb, cs + (c + 1) * 16);
                            tmem_ld_wait(p0);
                            tmem_ld16(taddr + (c + 1) * 16, p1);
                            promote16_cols(acc, c * 8, p0, rs2, csa);
                            if (c + 2 < NCH) load_cs(csa, cs + (c + 2) * 16);
                            tmem_ld_wait(p1);
                            if (c + 2 < NCH) tmem_ld16(taddr + (c + 2) * 16, p0);
                            promote16_cols(acc, (c + 1) * 8, p1, rs2, csb);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (kPair)
                        mbar_arrive_cluster_relaxed(tempty_remote[buf]);
                    else
                        mbar_arrive(&tempty_bar[buf]);
                    if (BASE == kWgrad) mbar_arrive(&sempty_bar[ss]);
                }
            }
            if (!ok) break;
            if ((kPair && !kGrp) || (kGrp && mo + quad * 32 + 31 < rlim)) {
                // Stage this warp's 32 rows x H columns (64-column boxes,
                // 128-byte swizzle: 16-byte chunk j of row r goes to j ^ (r % 8))
                // and hand them to the TMA; rows past R are clipped by it.  (A
                // grouped tile's warp whose rows cross its expert's end takes
                // the plain stores below instead.)
                const uint32_t wbuf = out_base + ew * CF::kOutWarpBytes;
                if constexpr (kStoreWarp) {
                    // the store warp has read out the previous tile's staging
                    if (!pwait(&sfree_bar, (tile_j & 1u) ^ 1u, SITE_GEMM_EPI_TMEM_FULL)) {
                        ok = false;
                        break;
                    }
                } else {
                    if (lane == 0) bulk_wait_group_read0();  // previous tile's stores have read it
                    __syncwarp();
                }
#pragma unroll
                for (int i = 0; i < H / 8; ++i) {
                    uint4 v;
                    v.x = pack_bf16x2(acc[4 * i + 0].x, acc[4 * i + 0].y);
                    v.y = pack_bf16x2(acc[4 * i + 1].x, acc[4 * i + 1].y);
                    v.z = pack_bf16x2(acc[4 * i + 2].x, acc[4 * i + 2].y);
                    v.w = pack_bf16x2(acc[4 * i + 3].x, acc[4 * i + 3].y);
                    const int half = i >> 3, chunk = i & 7;
                    const uint32_t a = wbuf + half * 4096 + lane * 128 + ((chunk ^ (lane & 7)) << 4);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x),
                                 "r"(v.y), "r"(v.z), "r"(v.w)
                                 : "memory");
                }
                fence_proxy_async();
                __syncwarp();
                if constexpr (kStoreWarp) {
                    if (lane == 0) mbar_arrive(&staged_bar);
                } else if (lane == 0) {
#pragma unroll
                    for (int h = 0; h < H / 64; ++h)
                        tma_store_2d_hint(&tmY, wbuf + 4096 * h, col0 + 64 * h, mo + quad * 32,
                                          pol_out);
                    bulk_commit_group();
                }
            } else if (splits > 1) {
                // FP32 partial of this contraction range (single-CTA kernel only)
                if (row_ok) {
                    const int sp = t % splits;
                    float4 *dst = reinterpret_cast<float4 *>(
                        partial + ((size_t)sp * R + row) * C + col0);
#pragma unroll
                    for (int i = 0; i < H / 4; ++i)
                        dst[i] = make_float4(acc[2 * i].x, acc[2 * i].y, acc[2 * i + 1].x,
                                             acc[2 * i + 1].y);
                }
            } else if (row_ok) {
                uint4 *dst = reinterpret_cast<uint4 *>(out + (size_t)row * C + col0);
#pragma unroll
                for (int i = 0; i < H / 8; ++i) {
                    uint4 v;
                    v.x = pack_bf16x2(acc[4 * i + 0].x, acc[4 * i + 0].y);
                    v.y = pack_bf16x2(acc[4 * i + 1].x, acc[4 * i + 1].y);
                    v.z = pack_bf16x2(acc[4 * i + 2].x, acc[4 * i + 2].y);
                    v.w = pack_bf16x2(acc[4 * i + 3].x, acc[4 * i + 3].y);
                    st_global_v4_hint(dst + i, v, pol_out);
                }
            }
        }
    }

    // Outstanding TMA stores must finish reading shared memory before exit.
    if ((kPair || kGrp) && warp >= 4 && (threadIdx.x & 31) == 0) bulk_wait_group0();
    tc_fence_before();
    // Neither CTA of a pair may exit or free TMEM while the other can still
    // use its barriers, shared memory or the pair's TMEM allocation.
    if (kPair)
        cluster_sync();
    else
        __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if (kPair)
            tmem_dealloc_pair(tmem, CF::kTmemCols);
        else
            tmem_dealloc(tmem, CF::kTmemCols);
    }
}

// out[i] = BF16(sum over sp = 0 .. splits-1 of partial[sp][i]), summed in that
// order; four elements per thread (R * C is a multiple of 128).  The partials
// are loaded eight splits at a time, so that a thread waits for one round
// trip per eight splits instead of one per split.
__global__ void __launch_bounds__(256)
splitk_reduce_kernel(const float4 *__restrict__ partial, int splits, int64_t n4,
                     uint2 *__restrict__ out) {
    griddep_launch_dependents();
    griddep_wait();
    constexpr int kB = 8;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
         i += (int64_t)gridDim.x * blockDim.x) {
        float4 a = partial[i];
        int sp = 1;
        for (; sp + kB <= splits; sp += kB) {
            float4 b[kB];
#pragma unroll
            for (int u = 0; u < kB; ++u) b[u] = partial[(int64_t)(sp + u) * n4 + i];
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                a.x += b[u].x;
                a.y += b[u].y;
                a.z += b[u].z;
                a.w += b[u].w;
            }
        }
        for (; sp < splits; ++sp) {
            const float4 b = partial[(int64_t)sp * n4 + i];
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
        }
        out[i] = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
    }
}

// Self-test of the bounded-wait path: waits on an mbarrier that nothing
// arrives at, so the wait gives up after `limit_cycles` and records a timeout.
__global__ void selftest_wait_kernel(unsigned *status, uint64_t limit_cycles) {
    __shared__ uint64_t bar;
    __shared__ volatile int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    mbar_wait(&bar, 0, &abort_flag, status, SITE_TEST_NEVER_SET, limit_cycles);
}

// ------------------------------------------------------------------- host --

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        cudaGetLastError();
    });
    return fn;
}

// Row-major BF16 matrix [outer][inner] for the pair kernel's output stores:
// box 32 rows x 64 columns (128 bytes), 128-byte swizzle.
bool make_map_out(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {64, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major uint8 matrix [outer][inner] with a box of box_outer x box_inner
// (box_inner = 128 bytes, 128-byte swizzle).
bool make_map_u8(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer,
                 uint32_t box_inner, uint32_t box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tile order.  An operand that the order walks again stays in L2 only while
// it takes at most kL2Budget bytes: measured on the 126 MB L2, a 33.5 MB
// operand walked by every tile row was read from DRAM once, a 58.7 MB one
// 4.8 to 6 times over (the outputs stream through L2 meanwhile).  So the
// smaller operand is kept whole when it fits.  Otherwise (long contractions)
// the tiles run in groups of at most 16 row tiles (mode 2) or column tiles
// (mode 3) whose operand fits, whichever reads fewer bytes in the model
// A + B x (row groups) or B + A x (column groups), column groups on a tie.
// Measured over every such product of the 8B and 32B training layers, the
// times of all reasonable orders lay within about 3% of each other; this
// one reads the fewest DRAM bytes of them (groups of 4 read up to 2.8x
// more), which matters under the power cap.  `rows` is the height of a row
// tile (BM x CL), `cols` the width of a column tile (BN).
Raster choose_raster(int64_t R, int64_t C, int64_t D, int64_t rows, int64_t cols) {
    const int64_t kL2Budget = 48ll << 20;
    constexpr int64_t kMaxGroup = 16;
    const int64_t a = R * D, b = C * D;
    if (a <= kL2Budget || b <= kL2Budget) return Raster{b <= a ? 0 : 1, 0};
    const int64_t tm = (R + rows - 1) / rows, tn = (C + cols - 1) / cols;
    // the fewest groups whose footprint fits, then groups of equal size
    auto groups = [&](int64_t tiles, int64_t tile_bytes, int64_t &per) {
        int64_t g = kL2Budget / tile_bytes;
        g = g < 1 ? 1 : (g > kMaxGroup ? kMaxGroup : g);
        const int64_t n = (tiles + g - 1) / g;
        per = (tiles + n - 1) / n;
        return n;
    };
    int64_t gm = 1, gn = 1;
    const int64_t nm = groups(tm, rows * D, gm), nn = groups(tn, cols * D, gn);
    if (a + b * nm < b + a * nn) return Raster{2, (int)gm};
    return Raster{3, (int)gn};
}

// Kernel arguments are passed by value; a CUtensorMap goes as is.
inline const CUtensorMap &tmA_arg(const CUtensorMap &m) { return m; }

template <int BN, int MODE, int CL, int ST = 0>
jet_status launch(const DeviceInfo &dev, const uint8_t *a, const float *sa, const uint8_t *b,
                  const float *sb, uint16_t *out, int64_t R, int64_t C, int64_t D, int splits,
                  float *partial, cudaStream_t stream, const int64_t *goff = nullptr,
                  int gE = 0, uint64_t wait_limit = kWaitLimitCycles) {
    using CF = Cfg<BN, CL, CL == 2 || is_grouped(MODE), ST>;
    auto kernel = gemm_fp8_kernel<BN, MODE, CL, ST>;
    static std::mutex mu;
    static int max_units[64] = {};  // co-resident CTAs (CL = 1) or clusters (CL = 2)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = CF::kSmemBytes;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic dependent launch (see launch_pdl); the occupancy query
    // below sees only the cluster attribute
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (max_units[dev.ordinal] == 0) {
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     CF::kSmemBytes) != cudaSuccess) {
                cudaGetLastError();
                return JET_ERR_CUDA;
            }
            int n = dev.num_sms / CL;
            if (CL > 1) {
                cfg.gridDim = dim3(dev.num_sms - dev.num_sms % CL);
                int clusters = 0;
                if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) == cudaSuccess &&
                    clusters > 0)
                    n = clusters;
                cudaGetLastError();
            }
            max_units[dev.ordinal] = n;
        }
    }
    CUtensorMap ta, tb, ty;
    if (!make_map_u8(&ta, a, (uint64_t)D, (uint64_t)R, BK, BM)) return JET_ERR_CUDA;
    constexpr int BASE = base_mode(MODE);
    constexpr bool kStagedOut = CL == 2 || is_grouped(MODE);
    // grouped WGrad writes the experts' dW stacked, [gE * R][C]
    const uint64_t out_rows = MODE == kWgradGrouped ? (uint64_t)gE * (uint64_t)R : (uint64_t)R;
    if (kStagedOut && !make_map_out(&ty, out, (uint64_t)C, out_rows)) return JET_ERR_CUDA;
    if (!kStagedOut) ty = ta;  // unused: this kernel stores from registers
    // grouped forward / DGrad: B is the experts' weights stacked, [gE * C][D]
    // (forward) or, read MN-major, [gE * D][C] (DGrad)
    const uint64_t b_rows = MODE == kFwdGrouped ? (uint64_t)gE * (uint64_t)C : (uint64_t)C;
    const uint64_t b_kdim = MODE == kDgradGrouped ? (uint64_t)gE * (uint64_t)D : (uint64_t)D;
    bool okb = BASE == kDgrad ? make_map_u8(&tb, b, (uint64_t)C, b_kdim, 128, BK)
                              : make_map_u8(&tb, b, (uint64_t)D, b_rows, BK, CF::kBRows);
    if (!okb) return JET_ERR_CUDA;
    // grouped forward / DGrad: at most one unit per expert more than the
    // dense count; grouped WGrad: every expert's whole dW
    const int64_t tiles_mn = (R + BM * CL - 1) / (BM * CL) * (C / BN);
    const int64_t units = MODE == kWgradGrouped ? gE * tiles_mn
                          : ((R + BM * CL - 1) / (BM * CL) + gE) * (C / BN) * splits;
    const int64_t grid_units = units < max_units[dev.ordinal] ? units : max_units[dev.ordinal];
    cfg.gridDim = dim3((unsigned)(grid_units * CL));
    const Raster raster = choose_raster(R, C, D, BM * CL, BN);
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kernel, tmA_arg(ta), tmA_arg(tb), tmA_arg(ty), sa, sb, out,
                           (int)R, (int)C, (int)D, raster, splits, partial, goff, gE,
                           dev.status_word, wait_limit) != cudaSuccess) {
        cudaGetLastError();
        return JET_ERR_CUDA;
    }
    if (splits > 1) {
        const int64_t n4 = R * C / 4;
        const int64_t want = (n4 + 255) / 256, cap = (int64_t)dev.num_sms * 8;
        return launch_pdl(splitk_reduce_kernel, dim3((unsigned)(want < cap ? want : cap)),
                          dim3(256), 0, stream, reinterpret_cast<const float4 *>(partial),
                          splits, n4, reinterpret_cast<uint2 *>(out));
    }
    return launch_status();
}

// How an R x C x D product of at most 512 rows (decode and short prefill) is
// cut.  Such a product has too few output tiles for 152 SMs; it runs on the
// single-CTA kernel with the contraction cut into ranges of whole
// 128-slices: about 128 units in all, at most 8 ranges per tile, at most one
// per slice, and FP32 partials (4 * splits * R * C bytes, written and read
// back by the reduction) of at most 32 MB, so that they stay in L2.  Tiles
// are 128 wide when that count is at least 2 (q, k, v, o and down of the 8B
// and 32B layers), else 256 wide (gate and up up to 128 rows); one range
// means no split (and rows above 128 then take the CTA-pair kernel).  A
// 128-wide unit of at least 8 slices on at most 64 rows, or of at least 24
// slices, runs on the six-stage kernel: there the weights stream from DRAM
// and the stages in flight set the rate, while on short units the larger
// shared-memory footprint cost 8-13% (k and v at 128-512 rows).  Measured on
// the 7 projections of both layers at 16 to 512 rows (weights streamed from
// DRAM): against 256-wide tiles throughout, 128-wide tiles took 12-38% less
// time on k and v at every row count and 10-30% on q, o and down at 32-256
// rows, and lost 10% on the 32B q at 16 rows; with fewer ranges per tile
// each unit runs a longer pipeline and the reduction reads fewer partials.
// The plan depends only on the sizes, never on the device, so the workspace
// size and the summation order (hence the result) are the same on every GPU.
constexpr int64_t kSplitMaxRows = 512;

struct SplitPlan {
    int splits;  // contraction ranges per output tile (1 = no split)
    int bn;      // tile width of a split product
    bool deep;   // six operand stages
};

int64_t split_count(int64_t R, int64_t C, int64_t D, int64_t bn) {
    constexpr int64_t kTargetUnits = 128, kMaxSplits = 8;
    constexpr int64_t kPartialBudget = 32ll << 20;
    const int64_t tiles = (R + BM - 1) / BM * (C / bn);
    int64_t s = kTargetUnits / tiles;
    if (s > kMaxSplits) s = kMaxSplits;
    if (s > D / BK) s = D / BK;
    while (s > 1 && 4 * s * R * C > kPartialBudget) --s;
    return s;
}

SplitPlan split_plan(int64_t R, int64_t C, int64_t D) {
    if (R <= 0 || R > kSplitMaxRows || C <= 0 || D <= 0 || C % 128 != 0 || D % BK != 0)
        return SplitPlan{1, 0, false};
    int64_t s = split_count(R, C, D, 128);
    if (s >= 2) {
        const int64_t slices = D / BK / s;
        return SplitPlan{(int)s, 128, (slices >= 8 && R <= 64) || slices >= 24};
    }
    if (C % 256 == 0 && (s = split_count(R, C, D, 256)) >= 2) return SplitPlan{(int)s, 256, false};
    return SplitPlan{1, 0, false};
}

int splitk_splits(int64_t R, int64_t C, int64_t D) { return split_plan(R, C, D).splits; }

size_t splitk_workspace(int64_t R, int64_t C, int64_t D) {
    const int s = splitk_splits(R, C, D);
    return s > 1 ? (size_t)s * (size_t)R * (size_t)C * sizeof(float) : 0;
}

template <int MODE>
jet_status run_gemm(const uint8_t *a, const float *sa, const uint8_t *b, const float *sb,
                    uint16_t *out, int64_t R, int64_t C, int64_t D, void *ws, jet_stream_t s) {
    DeviceInfo dev;
    jet_status st = current_device(&dev);
    if (st != JET_OK) return st;
    cudaStream_t stream = as_stream(s);
    if (R == 0 || C == 0) return JET_OK;
    if (D == 0) {  // empty contraction: the product is zero
        return cudaMemsetAsync(out, 0, (size_t)R * C * 2, stream) == cudaSuccess ? JET_OK
                                                                               : JET_ERR_CUDA;
    }
    // A split contraction runs on the single-CTA kernel (see split_plan);
    // otherwise the pair MMA (256 x 256 per CTA pair) whenever there are at
    // least two row tiles and the output is a multiple of 256 wide.
    const SplitPlan plan = MODE == kWgrad ? SplitPlan{1, 0, false} : split_plan(R, C, D);
    if (plan.splits > 1) {
        float *partial = static_cast<float *>(ws);
        if (plan.bn == 256)
            return launch<256, MODE, 1>(dev, a, sa, b, sb, out, R, C, D, plan.splits, partial,
                                        stream);
        if (plan.deep)
            return launch<128, MODE, 1, 6>(dev, a, sa, b, sb, out, R, C, D, plan.splits,
                                           partial, stream);
        return launch<128, MODE, 1>(dev, a, sa, b, sb, out, R, C, D, plan.splits, partial,
                                    stream);
    }
    if (C % 256 == 0) {
        if (R > BM) return launch<256, MODE, 2>(dev, a, sa, b, sb, out, R, C, D, 1, nullptr, stream);
        return launch<256, MODE, 1>(dev, a, sa, b, sb, out, R, C, D, 1, nullptr, stream);
    }
    return launch<128, MODE, 1>(dev, a, sa, b, sb, out, R, C, D, 1, nullptr, stream);
}

constexpr int64_t kMaxDim = (int64_t)1 << 30;

}  // namespace

// Forward products of one token, and of 2-4 tokens with M * N * K <= 2^25
// (e.g. two tokens on a 4096 x 4096 weight, four on 1024 x 4096), run on the
// CUDA-core kernel of gemv.cu (no workspace): its fixed cost per call is a
// fraction of the split tensor-core path's, and at one token it also streams
// the largest 8B weights faster; with more tokens its multiply-adds grow
// with M and the tensor path wins (measured on the 8B projections).
constexpr int64_t kGemvMaxRows = 4;
constexpr int64_t kGemvMaxMacs = (int64_t)1 << 25;
jet_status jet_gemv_fp8_fwd(const uint8_t *qx, const float *sx, const uint8_t *qw,
                            const float *sw, int64_t M, int64_t N, int64_t K, uint16_t *y,
                            int num_sms, cudaStream_t stream);
inline bool use_gemv(int64_t M, int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || M < 1 || M > kGemvMaxRows) return false;
    return M == 1 || M * N * K <= kGemvMaxMacs;
}

// Workspace bytes of a GEMM (JET_OP_GEMM_*), for jet_workspace_bytes().
size_t jet_gemm_workspace(int op, int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0) return 0;
    if (op == JET_OP_GEMM_FWD) return use_gemv(M, N, K) ? 0 : splitk_workspace(M, N, K);
    if (op == JET_OP_GEMM_DGRAD) return splitk_workspace(M, K, N);
    return 0;
}

extern "C" {

jet_status jet_gemm_fp8_fwd(const uint8_t *qx, const float *sx, const uint8_t *qw,
                            const float *sw, int64_t M, int64_t N, int64_t K, uint16_t *y,
                            void *ws, size_t ws_bytes, jet_stream_t stream) {
    JET_REQUIRE(M >= 0 && N >= 0 && K >= 0, JET_ERR_SHAPE);
    const bool out_empty = (M == 0 || N == 0), in_empty = out_empty || K == 0;
    JET_REQUIRE(out_empty || y, JET_ERR_NULL);
    JET_REQUIRE(in_empty || (qx && sx && qw && sw), JET_ERR_NULL);
    JET_REQUIRE(N % 128 == 0 && K % 128 == 0 && M < kMaxDim && N < kMaxDim && K < kMaxDim,
                JET_ERR_SHAPE);
    JET_REQUIRE(aligned16(qx) && aligned16(sx) && aligned16(qw) && aligned16(sw) &&
                    aligned16(y),
                JET_ERR_ALIGN);
    JET_REQUIRE(aligned16(ws), JET_ERR_ALIGN);
    const size_t need = jet_gemm_workspace(JET_OP_GEMM_FWD, M, N, K);
    JET_REQUIRE(need == 0 || (ws && ws_bytes >= need), JET_ERR_WORKSPACE);
    if (use_gemv(M, N, K)) {  // decode: weight streaming
        DeviceInfo dev;
        jet_status st = current_device(&dev);
        if (st != JET_OK) return st;
        return jet_gemv_fp8_fwd(qx, sx, qw, sw, M, N, K, y, dev.num_sms, as_stream(stream));
    }
    return run_gemm<kFwd>(qx, sx, qw, sw, y, M, N, K, ws, stream);
}

jet_status jet_gemm_fp8_fwd_grouped(const uint8_t *qx, const float *sx, const uint8_t *qw,
                                    const float *sw, const int64_t *offsets, int64_t E,
                                    int64_t M, int64_t N, int64_t K, uint16_t *y,
                                    jet_stream_t stream) {
    JET_REQUIRE(M >= 0 && N >= 0 && K >= 0 && E >= 1 && E <= kMaxGroups, JET_ERR_SHAPE);
    const bool out_empty = (M == 0 || N == 0), in_empty = out_empty || K == 0;
    JET_REQUIRE(out_empty || (y && offsets), JET_ERR_NULL);
    JET_REQUIRE(in_empty || (qx && sx && qw && sw), JET_ERR_NULL);
    JET_REQUIRE(N % 128 == 0 && K % 128 == 0 && M < kMaxDim && N < kMaxDim && K < kMaxDim &&
                    E * N < kMaxDim,
                JET_ERR_SHAPE);
    JET_REQUIRE(aligned16(qx) && aligned16(sx) && aligned16(qw) && aligned16(sw) &&
                    aligned16(offsets) && aligned16(y),
                JET_ERR_ALIGN);
    DeviceInfo dev;
    jet_status st = current_device(&dev);
    if (st != JET_OK) return st;
    cudaStream_t s = as_stream(stream);
    if (out_empty) return JET_OK;
    if (K == 0)  // empty contraction: the product is zero
        return cudaMemsetAsync(y, 0, (size_t)M * N * 2, s) == cudaSuccess ? JET_OK : JET_ERR_CUDA;
    if (N % 256 == 0)
        return launch<256, kFwdGrouped, 1>(dev, qx, sx, qw, sw, y, M, N, K, 1, nullptr, s, offsets,
                                           (int)E);
    return launch<128, kFwdGrouped, 1>(dev, qx, sx, qw, sw, y, M, N, K, 1, nullptr, s, offsets,
                                       (int)E);
}

jet_status jet_gemm_fp8_dgrad_grouped(const uint8_t *qdy, const float *sdy, const uint8_t *qw,
                                      const float *sw, const int64_t *offsets, int64_t E,
                                      int64_t M, int64_t N, int64_t K, uint16_t *dx,
                                      jet_stream_t stream) {
    JET_REQUIRE(M >= 0 && N >= 0 && K >= 0 && E >= 1 && E <= kMaxGroups, JET_ERR_SHAPE);
    const bool out_empty = (M == 0 || K == 0), in_empty = out_empty || N == 0;
    JET_REQUIRE(out_empty || (dx && offsets), JET_ERR_NULL);
    JET_REQUIRE(in_empty || (qdy && sdy && qw && sw), JET_ERR_NULL);
    JET_REQUIRE(N % 128 == 0 && K % 128 == 0 && M < kMaxDim && N < kMaxDim && K < kMaxDim &&
                    E * N < kMaxDim,
                JET_ERR_SHAPE);
    JET_REQUIRE(aligned16(qdy) && aligned16(sdy) && aligned16(qw) && aligned16(sw) &&
                    aligned16(offsets) && aligned16(dx),
                JET_ERR_ALIGN);
    DeviceInfo dev;
    jet_status st = current_device(&dev);
    if (st != JET_OK) return st;
    cudaStream_t s = as_stream(stream);
    if (out_empty) return JET_OK;
    if (N == 0)  // empty contraction: the product is zero
        return cudaMemsetAsync(dx, 0, (size_t)M * K * 2, s) == cudaSuccess ? JET_OK : JET_ERR_CUDA;
    // rows R = tokens, columns C = K, contraction D = N
    if (K % 256 == 0)
        return launch<256, kDgradGrouped, 1>(dev, qdy, sdy, qw, sw, dx, M, K, N, 1, nullptr, s,
                                             offsets, (int)E);
    return launch<128, kDgradGrouped, 1>(dev, qdy, sdy, qw, sw, dx, M, K, N, 1, nullptr, s,
                                         offsets, (int)E);
}

jet_status jet_gemm_fp8_wgrad_grouped(const uint8_t *qdyT, const float *sdyT, const uint8_t *qxT,
                                      const float *sxT, const int64_t *offsets, int64_t E,
                                      int64_t M, int64_t N, int64_t K, uint16_t *dw,
                                      jet_stream_t stream) {
    JET_REQUIRE(M >= 0 && N >= 0 && K >= 0 && E >= 1 && E <= kMaxGroups, JET_ERR_SHAPE);
    const bool out_empty = (N == 0 || K == 0), in_empty = out_empty || M == 0;
    JET_REQUIRE(out_empty || (dw && offsets), JET_ERR_NULL);
    JET_REQUIRE(in_empty || (qdyT && sdyT && qxT && sxT), JET_ERR_NULL);
    JET_REQUIRE(M % 128 == 0 && N % 128 == 0 && K % 128 == 0 && M < kMaxDim && N < kMaxDim &&
                    K < kMaxDim && E * N < kMaxDim,
                JET_ERR_SHAPE);
    JET_REQUIRE(aligned16(qdyT) && aligned16(sdyT) && aligned16(qxT) && aligned16(sxT) &&
                    aligned16(offsets) && aligned16(dw),
                JET_ERR_ALIGN);
    DeviceInfo dev;
    jet_status st = current_device(&dev);
    if (st != JET_OK) return st;
    cudaStream_t s = as_stream(stream);
    if (out_empty) return JET_OK;
    if (M == 0)  // no tokens: every expert's gradient is zero
        return cudaMemsetAsync(dw, 0, (size_t)E * N * K * 2, s) == cudaSuccess ? JET_OK
                                                                             : JET_ERR_CUDA;
    // rows R = N (per expert), columns C = K, contraction D = M (the expert's
    // token blocks); CTA pairs over 256 rows of an expert's dW when K is a
    // multiple of 256 and N has at least two row tiles
    if (K % 256 == 0) {
        if (N > BM)
            return launch<256, kWgradGrouped, 2>(dev, qdyT, sdyT, qxT, sxT, dw, N, K, M, 1,
                                                 nullptr, s, offsets, (int)E);
        return launch<256, kWgradGrouped, 1>(dev, qdyT, sdyT, qxT, sxT, dw, N, K, M, 1, nullptr,
                                             s, offsets, (int)E);
    }
    return launch<128, kWgradGrouped, 1>(dev, qdyT, sdyT, qxT, sxT, dw, N, K, M, 1, nullptr, s,
                                         offsets, (int)E);
}

jet_status jet_gemm_fp8_dgrad(const uint8_t *qdy, const float *sdy, const uint8_t *qw,
                              const float *sw, int64_t M, int64_t N, int64_t K, uint16_t *dx,
                              void *ws, size_t ws_bytes, jet_stream_t stream) {
    JET_REQUIRE(M >= 0 && N >= 0 && K >= 0, JET_ERR_SHAPE);
    const bool out_empty = (M == 0 || K == 0), in_empty = out_empty || N == 0;
    JET_REQUIRE(out_empty || dx, JET_ERR_NULL);
    JET_REQUIRE(in_empty || (qdy && sdy && qw && sw), JET_ERR_NULL);
    JET_REQUIRE(N % 128 == 0 && K % 128 == 0 && M < kMaxDim && N < kMaxDim && K < kMaxDim,
                JET_ERR_SHAPE);
    JET_REQUIRE(aligned16(qdy) && aligned16(sdy) && aligned16(qw) && aligned16(sw) &&
                    aligned16(dx),
                JET_ERR_ALIGN);
    JET_REQUIRE(aligned16(ws), JET_ERR_ALIGN);
    const size_t need = splitk_workspace(M, K, N);
    JET_REQUIRE(need == 0 || (ws && ws_bytes >= need), JET_ERR_WORKSPACE);
    return run_gemm<kDgrad>(qdy, sdy, qw, sw, dx, M, K, N, ws, stream);
}

jet_status jet_gemm_fp8_wgrad(const uint8_t *qdyT, const float *sdyT, const uint8_t *qxT,
                              const float *sxT, int64_t M, int64_t N, int64_t K, uint16_t *dw,
                              void *ws, size_t ws_bytes, jet_stream_t stream) {
    (void)ws_bytes;
    JET_REQUIRE(M >= 0 && N >= 0 && K >= 0, JET_ERR_SHAPE);
    const bool out_empty = (N == 0 || K == 0), in_empty = out_empty || M == 0;
    JET_REQUIRE(out_empty || dw, JET_ERR_NULL);
    JET_REQUIRE(in_empty || (qdyT && sdyT && qxT && sxT), JET_ERR_NULL);
    JET_REQUIRE(M % 128 == 0 && N % 128 == 0 && K % 128 == 0 && M < kMaxDim && N < kMaxDim &&
                    K < kMaxDim,
                JET_ERR_SHAPE);
    JET_REQUIRE(aligned16(qdyT) && aligned16(sdyT) && aligned16(qxT) && aligned16(sxT) &&
                    aligned16(dw),
                JET_ERR_ALIGN);
    return run_gemm<kWgrad>(qdyT, sdyT, qxT, sxT, dw, N, K, M, ws, stream);
}

jet_status jet_selftest_gemm_timeout(const uint8_t *qx, const float *sx, const uint8_t *qw,
                                     const float *sw, int64_t M, int64_t N, int64_t K,
                                     uint16_t *y, uint64_t limit_cycles, jet_stream_t stream) {
    JET_REQUIRE(qx && sx && qw && sw && y, JET_ERR_NULL);
    JET_REQUIRE(M >= 1 && M <= BM && N >= 128 && K >= 128 && N % 128 == 0 && K % 128 == 0 &&
                    N < kMaxDim && K < kMaxDim,
                JET_ERR_SHAPE);
    JET_REQUIRE(limit_cycles >= 1 && limit_cycles <= kWaitLimitCycles, JET_ERR_SHAPE);
    JET_REQUIRE(aligned16(qx) && aligned16(sx) && aligned16(qw) && aligned16(sw) &&
                    aligned16(y),
                JET_ERR_ALIGN);
    DeviceInfo dev;
    jet_status st = current_device(&dev);
    if (st != JET_OK) return st;
    // the single-CTA forward kernel, contraction not split
    if (N % 256 == 0)
        return launch<256, kFwdTimeoutTest, 1>(dev, qx, sx, qw, sw, y, M, N, K, 1, nullptr,
                                               as_stream(stream), nullptr, 0, limit_cycles);
    return launch<128, kFwdTimeoutTest, 1>(dev, qx, sx, qw, sw, y, M, N, K, 1, nullptr,
                                           as_stream(stream), nullptr, 0, limit_cycles);
}

jet_status jet_selftest_bounded_wait(uint32_t limit_us, jet_stream_t stream) {
    JET_REQUIRE(limit_us >= 1 && limit_us <= 1000000u, JET_ERR_SHAPE);
    DeviceInfo dev;
    jet_status st = current_device(&dev);
    if (st != JET_OK) return st;
    // limit in SM cycles at the 2.07 GHz maximum clock (longer at lower clocks)
    selftest_wait_kernel<<<1, 32, 0, as_stream(stream)>>>(dev.status_word,
                                                          (uint64_t)limit_us * 2070ull);
    return launch_status();
}

}  // extern "C"
