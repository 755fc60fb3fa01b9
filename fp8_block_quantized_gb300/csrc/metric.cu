// token-mult-prob-error = (1/n) * sum_i exp(|logp_train_i - logp_rollout_i|)
// ("NVIDIA强化学习加速实操：10分钟提升2倍训练效率", section
// "FP8面临的关键挑战：数值分歧").  Two passes: a grid of G blocks streams the two
// FP32 vectors with 16-byte loads (each thread issues the loads of kUnroll
// grid strides before using them, so its share of the vectors is in flight
// at once rather than one round trip per stride; the order of its sums is
// the stride order either way), sums exp|a-b| in FP32 per thread and in
// FP64 across the block, and stores one FP64 partial per block in the
// workspace; one block then adds the G partials in a fixed order (so the
// result is deterministic) and writes the mean as FP32.
#include <mutex>

#include "jet_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kMaxBlocks = 1024;
constexpr int64_t kElemsPerBlockTarget = 2048;
constexpr int kUnroll = 4;  // grid strides whose loads a thread issues together

__device__ __forceinline__ float4 ld_stream_f4(const float *p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// FP64 sum over the block (the second passes, one block each).
__device__ __forceinline__ double block_sum(double v) {
    __shared__ double warp_sum[kThreads / 32];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = v;
    __syncthreads();
    double t = 0.0;
    if (threadIdx.x == 0)
        for (int i = 0; i < kThreads / 32; ++i) t += warp_sum[i];
    return t;  // valid in thread 0
}

// Sum over the block of one FP32 value per thread (the first passes, run by
// every block): a butterfly over each warp in FP32 (every lane ends with the
// same bits, additions being commutative), then the warps' sums in FP64 by
// thread 0 in warp order.  FP64 arithmetic is scarce on this GPU: the same
// tree in FP64 on every thread took about 40% of the per-sequence pass.  The
// FP32 tree adds at most 5 roundings (under 3.1e-7 relative) to a sum of
// positive terms.
__device__ __forceinline__ double block_sum_f(float v) {
    __shared__ double warp_sum[kThreads / 32];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = (double)v;
    __syncthreads();
    double t = 0.0;
    if (threadIdx.x == 0)
        for (int i = 0; i < kThreads / 32; ++i) t += warp_sum[i];
    return t;  // valid in thread 0
}

// Exact integer sum over the block (token counts).
__device__ __forceinline__ long long block_count(int c) {
    __shared__ long long warp_cnt[kThreads / 32];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
    if ((threadIdx.x & 31) == 0) warp_cnt[threadIdx.x >> 5] = c;
    __syncthreads();
    long long t = 0;
    if (threadIdx.x == 0)
        for (int i = 0; i < kThreads / 32; ++i) t += warp_cnt[i];
    return t;  // valid in thread 0
}

__global__ void __launch_bounds__(kThreads)
tmpe_partial_kernel(const float *__restrict__ a, const float *__restrict__ b, int64_t n,
                    double *__restrict__ partial) {
    jet::griddep_launch_dependents();
    jet::griddep_wait();
    float acc = 0.0f;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    const int64_t n4 = n >> 2;
    for (int64_t i0 = tid; i0 < n4; i0 += stride * kUnroll) {
        float4 x[kUnroll], y[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            x[u] = y[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (i < n4) {
                x[u] = ld_stream_f4(a + 4 * i);
                y[u] = ld_stream_f4(b + 4 * i);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (i0 + u * stride < n4) {
                acc += expf(fabsf(x[u].x - y[u].x));
                acc += expf(fabsf(x[u].y - y[u].y));
                acc += expf(fabsf(x[u].z - y[u].z));
                acc += expf(fabsf(x[u].w - y[u].w));
            }
        }
    }
    for (int64_t i = 4 * n4 + tid; i < n; i += stride) acc += expf(fabsf(a[i] - b[i]));
    const double t = block_sum_f(acc);
    if (threadIdx.x == 0) partial[blockIdx.x] = t;
}

__global__ void __launch_bounds__(kThreads)
tmpe_final_kernel(const double *__restrict__ partial, int nblocks, int64_t n, float *out) {
    jet::griddep_launch_dependents();
    jet::griddep_wait();
    double v = 0.0;
    for (int i = threadIdx.x; i < nblocks; i += kThreads) v += partial[i];
    const double t = block_sum(v);
    if (threadIdx.x == 0) *out = (float)(t / (double)n);
}

}  // namespace

int jet_metric_blocks(int64_t n) {
    int64_t g = (n + kElemsPerBlockTarget - 1) / kElemsPerBlockTarget;
    if (g < 1) g = 1;
    if (g > kMaxBlocks) g = kMaxBlocks;
    return (int)g;
}

// Launches both passes with `partial` (>= jet_metric_blocks(n) doubles) as the
// scratch array; arguments already validated.
jet_status jet_metric_launch(const float *a, const float *b, int64_t n, float *out,
                             double *partial, cudaStream_t stream) {
    const int g = jet_metric_blocks(n);
    jet_status st = jet::launch_pdl(tmpe_partial_kernel, dim3(g), dim3(kThreads), 0, stream, a, b,
                                    n, partial);
    if (st != JET_OK) return st;
    return jet::launch_pdl(tmpe_final_kernel, dim3(1), dim3(kThreads), 0, stream,
                           static_cast<const double *>(partial), g, n, out);
}

extern "C" jet_status jet_token_mult_prob_error(const float *logp_train,
                                                const float *logp_rollout, int64_t n,
                                                float *out, void *ws, size_t ws_bytes,
                                                jet_stream_t stream) {
    JET_REQUIRE(logp_train && logp_rollout && out, JET_ERR_NULL);
    JET_REQUIRE(n >= 1, JET_ERR_SHAPE);
    JET_REQUIRE(jet::aligned16(logp_train) && jet::aligned16(logp_rollout) &&
                    jet::aligned16(out) && jet::aligned16(ws),
                JET_ERR_ALIGN);
    const size_t need = (size_t)jet_metric_blocks(n) * sizeof(double);
    JET_REQUIRE(ws != nullptr && ws_bytes >= need, JET_ERR_WORKSPACE);
    jet::DeviceInfo dev;
    jet_status st = jet::current_device(&dev);
    if (st != JET_OK) return st;
    return jet_metric_launch(logp_train, logp_rollout, n, out, static_cast<double *>(ws),
                             jet::as_stream(stream));
}

// ---------------------------------------------------------------------------
// Variant that allocates nothing: the per-block partial sums live in a
// file-scope device array instead of a caller-supplied workspace.
// ---------------------------------------------------------------------------

namespace {

// Capacity of the static scratch: one FP64 partial per first-pass block.
constexpr int kNoAllocPartials = 1024;
// Largest n this variant accepts: the first pass uses one block per 2048
// tokens, so 1024 partials cover 2,097,152 tokens.
constexpr int64_t kNoAllocMaxTokens = (int64_t)kNoAllocPartials * kElemsPerBlockTarget;

// 8 KB on every device that loads the library, kept until the process exits
// (or until the device is reset, after which it is loaded again).
// In host code this name is only a host-side stand-in for the device array;
// its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) double g_tmpe_scratch[kNoAllocPartials];

std::mutex g_scratch_mu;
struct ScratchAddr {
    double *ptr;
    void *context;  // the context the address was looked up in
};
ScratchAddr g_scratch[64] = {};

// Device address of g_tmpe_scratch on the current device `dev` (with that
// device current), looked up on the first call in each context and cached:
// after a device reset the module is loaded again and the array may move, so
// a cached address is only reused while the context is the same.
jet_status scratch_address(const jet::DeviceInfo &dev, double **out) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (dev.ordinal < 0 || dev.ordinal >= 64) return JET_ERR_DEVICE;
    ScratchAddr &c = g_scratch[dev.ordinal];
    if (c.ptr == nullptr || c.context != dev.context) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_tmpe_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return JET_ERR_CUDA;
        }
        c.ptr = static_cast<double *>(p);
        c.context = dev.context;
    }
    *out = c.ptr;
    return JET_OK;
}

}  // namespace

extern "C" jet_status jet_token_mult_prob_error_noalloc(const float *logp_train,
                                                        const float *logp_rollout, int64_t n,
                                                        float *out, jet_stream_t stream) {
    JET_REQUIRE(logp_train && logp_rollout && out, JET_ERR_NULL);
    JET_REQUIRE(n >= 1 && n <= kNoAllocMaxTokens, JET_ERR_SHAPE);
    JET_REQUIRE(jet::aligned16(logp_train) && jet::aligned16(logp_rollout) &&
                    jet::aligned16(out),
                JET_ERR_ALIGN);
    jet::DeviceInfo dev;
    jet_status st = jet::current_device(&dev);
    if (st != JET_OK) return st;
    if (jet_metric_blocks(n) > kNoAllocPartials) return JET_ERR_SHAPE;
    double *partial = nullptr;
    st = scratch_address(dev, &partial);
    if (st != JET_OK) return st;
    // Every slot the second pass reads is written by the first pass of this
    // call, so the array needs no clearing between calls.
    return jet_metric_launch(logp_train, logp_rollout, n, out, partial, jet::as_stream(stream));
}

// ---------------------------------------------------------------------------
// Masked metric with per-token importance weights, one pass over the tokens.
// The importance weight of a token is the ratio of the training model's
// probability of it to the rollout model's ("FP8-RL" article: the ratio of
// the original to the compressed model's token probability; nmedialink page,
// section "重要抽样技术：提升RL精度的尖兵"): w_i = exp(a_i - b_i) with
// a = logp_train, b = logp_rollout, capped at `cap` when cap > 0 (the pages
// give no constant), 0 outside the mask.  The metric is token-mult-prob-error
// over the masked tokens.  Pass 1: four tokens per thread and step (16-byte
// loads of a and b, one 4-byte load of the mask, a 16-byte store of w; the
// loads of kUnroll steps issued together), FP32 sums per thread, FP64 per
// block; pass 2 adds the block partials in order.
// ---------------------------------------------------------------------------

namespace {

__device__ __forceinline__ float is_weight(float d, float cap) {
    const float w = expf(d);
    return cap > 0.0f ? fminf(w, cap) : w;
}

__global__ void __launch_bounds__(kThreads)
tmm_partial_kernel(const float *__restrict__ a, const float *__restrict__ b,
                   const uint8_t *__restrict__ mask, int64_t n, float cap,
                   float *__restrict__ w, double *__restrict__ partial) {
    jet::griddep_launch_dependents();
    jet::griddep_wait();
    float acc = 0.0f;
    int cnt = 0;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    const int64_t n4 = n >> 2;
    for (int64_t i0 = tid; i0 < n4; i0 += stride * kUnroll) {
        float4 x[kUnroll], y[kUnroll];
        uint32_t m4[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            x[u] = y[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            m4[u] = 0u;
            if (i < n4) {
                x[u] = ld_stream_f4(a + 4 * i);
                y[u] = ld_stream_f4(b + 4 * i);
                m4[u] = mask ? *reinterpret_cast<const uint32_t *>(mask + 4 * i) : 0x01010101u;
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            if (i >= n4) continue;
            const float d[4] = {x[u].x - y[u].x, x[u].y - y[u].y, x[u].z - y[u].z,
                                x[u].w - y[u].w};
            float wv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool on = ((m4[u] >> (8 * j)) & 0xFFu) != 0u;
                wv[j] = on ? is_weight(d[j], cap) : 0.0f;
                acc += on ? expf(fabsf(d[j])) : 0.0f;
                cnt += on ? 1 : 0;
            }
            if (w) *reinterpret_cast<float4 *>(w + 4 * i) = make_float4(wv[0], wv[1], wv[2], wv[3]);
        }
    }
    for (int64_t i = 4 * n4 + tid; i < n; i += stride) {
        const bool on = mask == nullptr || mask[i] != 0;
        const float d = a[i] - b[i];
        if (w) w[i] = on ? is_weight(d, cap) : 0.0f;
        acc += on ? expf(fabsf(d)) : 0.0f;
        cnt += on ? 1 : 0;
    }
    const double t = block_sum_f(acc);
    const long long c = block_count(cnt);
    if (threadIdx.x == 0) {
        partial[2 * blockIdx.x] = t;
        partial[2 * blockIdx.x + 1] = (double)c;
    }
}

__global__ void __launch_bounds__(kThreads)
tmm_final_kernel(const double *__restrict__ partial, int nblocks, float *out, int64_t *count) {
    jet::griddep_launch_dependents();
    jet::griddep_wait();
    double v = 0.0, c = 0.0;
    for (int i = threadIdx.x; i < nblocks; i += kThreads) {
        v += partial[2 * i];
        c += partial[2 * i + 1];
    }
    const double t = block_sum(v);
    __syncthreads();
    const double tc = block_sum(c);
    if (threadIdx.x == 0) {
        *out = tc > 0.0 ? (float)(t / tc) : __int_as_float(0x7fc00000);  // NaN: no masked token
        if (count) *count = (int64_t)tc;
    }
}

}  // namespace

namespace {

// Per-sequence variant: one block of 256 threads per sequence (a long
// sequence is streamed by 256 threads rather than one warp; one block per
// sequence, not a grid-stride loop over them, so that the hardware starts a
// block wherever one has finished and the uneven lengths balance
// themselves), threads striding over the sequence's tokens eight at a time
// (all loads of a step issued before use: the longest sequence sets the
// kernel's time, one round trip to memory per step); exp|a-b| of a step's
// tokens summed in FP32, the steps in FP64; the block's sums combined in a
// fixed order (deterministic).  Measured on 2048 log-normal sequences over
// 4 M tokens: 35.5 us, against 39.6 for a grid of 8 blocks per SM striding
// over the sequences with 4 tokens per step, 52.9 with 2 tokens per step,
// and 60-124 us for 512- or 1024-thread blocks.
constexpr int kSeqUnroll = 8;

__global__ void __launch_bounds__(kThreads)
tms_kernel(const float *__restrict__ a, const float *__restrict__ b,
           const uint8_t *__restrict__ mask, const int64_t *__restrict__ off, int64_t S,
           int64_t n, float cap, float *__restrict__ w, float *__restrict__ out,
           int64_t *__restrict__ count) {
    jet::griddep_launch_dependents();
    jet::griddep_wait();
    auto clampn = [&](int64_t v) { return v < 0 ? (int64_t)0 : (v > n ? n : v); };
    for (int64_t s = blockIdx.x; s < S; s += gridDim.x) {
        const int64_t lo = clampn(off[s]);
        const int64_t hi = max(lo, clampn(off[s + 1]));
        double sum = 0.0;
        int cnt = 0;
        for (int64_t i0 = lo + threadIdx.x; i0 < hi; i0 += (int64_t)kThreads * kSeqUnroll) {
            float x[kSeqUnroll], y[kSeqUnroll];
            bool on[kSeqUnroll];
#pragma unroll
            for (int u = 0; u < kSeqUnroll; ++u) {
                const int64_t i = i0 + (int64_t)kThreads * u;
                const bool in = i < hi;
                x[u] = in ? a[i] : 0.0f;
                y[u] = in ? b[i] : 0.0f;
                on[u] = in && (mask == nullptr || mask[i] != 0);
            }
            float part = 0.0f;
#pragma unroll
            for (int u = 0; u < kSeqUnroll; ++u) {
                const int64_t i = i0 + (int64_t)kThreads * u;
                const float d = x[u] - y[u];
                if (w && i < hi) w[i] = on[u] ? is_weight(d, cap) : 0.0f;
                part += on[u] ? expf(fabsf(d)) : 0.0f;
                cnt += on[u] ? 1 : 0;
            }
            sum += (double)part;
        }
        const double t = block_sum_f((float)sum);
        const long long c = block_count(cnt);
        if (threadIdx.x == 0) {
            out[s] = c > 0 ? (float)(t / (double)c) : __int_as_float(0x7fc00000);
            if (count) count[s] = (int64_t)c;
        }
        __syncthreads();  // before the next sequence reuses the scratch
    }
}

}  // namespace

extern "C" jet_status jet_token_mismatch_per_sequence(
    const float *logp_train, const float *logp_rollout, const uint8_t *mask,
    const int64_t *seq_offsets, int64_t S, int64_t n, float cap, float *w, float *out,
    int64_t *count, jet_stream_t stream) {
    JET_REQUIRE(S >= 1 && n >= 0, JET_ERR_SHAPE);
    JET_REQUIRE(seq_offsets && out && (n == 0 || (logp_train && logp_rollout)), JET_ERR_NULL);
    JET_REQUIRE(jet::aligned16(logp_train) && jet::aligned16(logp_rollout) &&
                    jet::aligned16(mask) && jet::aligned16(seq_offsets) && jet::aligned16(w) &&
                    jet::aligned16(out) && jet::aligned16(count),
                JET_ERR_ALIGN);
    jet::DeviceInfo dev;
    jet_status st = jet::current_device(&dev);
    if (st != JET_OK) return st;
    // one block per sequence, within the grid's limit (the kernel strides
    // over sequences beyond it)
    const int64_t cap_blocks = (int64_t)1 << 30;
    return jet::launch_pdl(tms_kernel, dim3((unsigned)(S < cap_blocks ? S : cap_blocks)),
                           dim3(kThreads), 0, jet::as_stream(stream), logp_train, logp_rollout,
                           mask, seq_offsets, S, n, cap, w, out, count);
}

// Workspace of jet_token_mismatch_masked: a sum and a count per first-pass block.
size_t jet_mismatch_masked_workspace(int64_t n) {
    return n > 0 ? (size_t)jet_metric_blocks(n) * 2 * sizeof(double) : 0;
}

extern "C" jet_status jet_token_mismatch_masked(const float *logp_train, const float *logp_rollout,
                                                const uint8_t *mask, int64_t n, float cap,
                                                float *w, float *out, int64_t *count, void *ws,
                                                size_t ws_bytes, jet_stream_t stream) {
    JET_REQUIRE(logp_train && logp_rollout && out, JET_ERR_NULL);
    JET_REQUIRE(n >= 1, JET_ERR_SHAPE);
    JET_REQUIRE(jet::aligned16(logp_train) && jet::aligned16(logp_rollout) &&
                    jet::aligned16(mask) && jet::aligned16(w) && jet::aligned16(out) &&
                    jet::aligned16(count) && jet::aligned16(ws),
                JET_ERR_ALIGN);
    JET_REQUIRE(ws != nullptr && ws_bytes >= jet_mismatch_masked_workspace(n), JET_ERR_WORKSPACE);
    jet::DeviceInfo dev;
    jet_status st = jet::current_device(&dev);
    if (st != JET_OK) return st;
    const int g = jet_metric_blocks(n);
    double *partial = static_cast<double *>(ws);
    cudaStream_t s = jet::as_stream(stream);
    st = jet::launch_pdl(tmm_partial_kernel, dim3(g), dim3(kThreads), 0, s, logp_train,
                         logp_rollout, mask, n, cap, w, partial);
    if (st != JET_OK) return st;
    return jet::launch_pdl(tmm_final_kernel, dim3(1), dim3(kThreads), 0, s,
                           static_cast<const double *>(partial), g, out, count);
}
