// token-mult-prob-error = (1/n) * sum_i exp(|logp_train_i - logp_rollout_i|)
// ("NVIDIA强化学习加速实操：10分钟提升2倍训练效率", section
// "FP8面临的关键挑战：数值分歧").  Two passes: a grid of G blocks streams the two
// FP32 vectors with 16-byte loads, sums exp|a-b| in FP32 per thread and in
// FP64 across the block, and stores one FP64 partial per block in the
// workspace; one block then adds the G partials in a fixed order (so the
// result is deterministic) and writes the mean as FP32.
#include <mutex>

#include "jet_common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kMaxBlocks = 1024;
constexpr int64_t kElemsPerBlockTarget = 2048;

__device__ __forceinline__ float4 ld_stream_f4(const float *p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

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

__global__ void __launch_bounds__(kThreads)
tmpe_partial_kernel(const float *__restrict__ a, const float *__restrict__ b, int64_t n,
                    double *__restrict__ partial) {
    jet::griddep_launch_dependents();
    jet::griddep_wait();
    float acc = 0.0f;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    const int64_t n4 = n >> 2;
    for (int64_t i = tid; i < n4; i += stride) {
        const float4 x = ld_stream_f4(a + 4 * i);
        const float4 y = ld_stream_f4(b + 4 * i);
        acc += expf(fabsf(x.x - y.x));
        acc += expf(fabsf(x.y - y.y));
        acc += expf(fabsf(x.z - y.z));
        acc += expf(fabsf(x.w - y.w));
    }
    for (int64_t i = 4 * n4 + tid; i < n; i += stride) acc += expf(fabsf(a[i] - b[i]));
    const double t = block_sum((double)acc);
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

// 8 KB on every device that loads the library, kept until the process exits.
// In host code this name is only a host-side stand-in for the device array;
// its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) double g_tmpe_scratch[kNoAllocPartials];

std::mutex g_scratch_mu;
double *g_scratch_ptr[64] = {};

// Device address of g_tmpe_scratch on the current device `dev`, looked up once
// per device (with that device current) and cached.
jet_status scratch_address(int dev, double **out) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (dev < 0 || dev >= 64) return JET_ERR_DEVICE;
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_tmpe_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return JET_ERR_CUDA;
        }
        g_scratch_ptr[dev] = static_cast<double *>(p);
    }
    *out = g_scratch_ptr[dev];
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
    st = scratch_address(dev.ordinal, &partial);
    if (st != JET_OK) return st;
    // Every slot the second pass reads is written by the first pass of this
    // call, so the array needs no clearing between calls.
    return jet_metric_launch(logp_train, logp_rollout, n, out, partial, jet::as_stream(stream));
}
