// Library-wide entry points: status strings, device checks, the device-side
// status word and workspace sizing.
#include <cuda.h>

#include <mutex>

#include "jet_common.cuh"

// Device-side status word: kernels record bounded-wait timeouts here.
__device__ unsigned g_jet_status_word;

namespace jet {

namespace {
constexpr int kMaxDevices = 64;
struct Cached {
    int state;  // 0 unknown, 1 ok, 2 wrong arch
    int num_sms;
    unsigned *status_word;
    void *context;  // the context the status word's address belongs to
};
Cached g_cache[kMaxDevices];
std::mutex g_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
        cudaGetLastError();
    });
    return fn;
}
}  // namespace

void *current_context() {
    CtxGetCurrentFn fn = ctx_get_current_fn();
    CUcontext ctx = nullptr;
    if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
    return static_cast<void *>(ctx);
}

jet_status current_device(DeviceInfo *info) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return JET_ERR_DEVICE;
    }
    // After cudaDeviceReset (or any other teardown of the device's primary
    // context) the module is loaded again and a __device__ variable can sit at
    // a new address, so the cached address is only trusted for the context it
    // was looked up in.
    void *ctx = current_context();
    std::lock_guard<std::mutex> lock(g_mu);
    Cached &c = g_cache[dev];
    if (c.state == 1 && c.context != ctx) c.state = 0;
    if (c.state == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return JET_ERR_DEVICE;
        }
        if (major != 10 || minor != 3) {
            c.state = 2;
        } else {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_jet_status_word) != cudaSuccess) {
                cudaGetLastError();
                return JET_ERR_CUDA;
            }
            // the lookup may have created the primary context: ask again
            if (ctx == nullptr) ctx = current_context();
            c.num_sms = sms;
            c.status_word = static_cast<unsigned *>(p);
            c.context = ctx;
            c.state = 1;
        }
    }
    if (c.state != 1) return JET_ERR_DEVICE;
    info->ordinal = dev;
    info->num_sms = c.num_sms;
    info->status_word = c.status_word;
    info->context = ctx;
    return JET_OK;
}

}  // namespace jet

// Size of the per-block partial-sum array of the metric's first pass.
int jet_metric_blocks(int64_t n);
// FP32 partial tiles of a split-contraction GEMM (0 when it is not split).
size_t jet_gemm_workspace(int op, int64_t M, int64_t N, int64_t K);
// Per-block sums and counts of the masked metric's first pass.
size_t jet_mismatch_masked_workspace(int64_t n);

extern "C" {

const char *jet_status_str(int status) {
    switch (status) {
    case JET_OK: return "JET_OK";
    case JET_ERR_NULL: return "JET_ERR_NULL";
    case JET_ERR_SHAPE: return "JET_ERR_SHAPE";
    case JET_ERR_ALIGN: return "JET_ERR_ALIGN";
    case JET_ERR_CUDA: return "JET_ERR_CUDA";
    case JET_ERR_DEVICE: return "JET_ERR_DEVICE";
    case JET_ERR_WORKSPACE: return "JET_ERR_WORKSPACE";
    case JET_ERR_TIMEOUT: return "JET_ERR_TIMEOUT";
    default: return "JET_ERR_UNKNOWN";
    }
}

int jet_version(void) { return 10000; }

size_t jet_workspace_bytes(int op, int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0) return 0;
    switch (op) {
    case JET_OP_TOKEN_MULT_PROB_ERROR:
        return M > 0 ? (size_t)jet_metric_blocks(M) * sizeof(double) : 0;
    case JET_OP_GEMM_FWD:
    case JET_OP_GEMM_DGRAD:
        return jet_gemm_workspace(op, M, N, K);
    case JET_OP_TOKEN_MISMATCH_MASKED:
        return jet_mismatch_masked_workspace(M);
    default:
        return 0;
    }
}

jet_status jet_device_status(jet_stream_t stream, uint32_t *detail) {
    if (detail) *detail = 0;
    jet::DeviceInfo info;
    jet_status st = jet::current_device(&info);
    if (st != JET_OK) return st;
    if (cudaStreamSynchronize(jet::as_stream(stream)) != cudaSuccess) {
        cudaGetLastError();
        return JET_ERR_CUDA;
    }
    unsigned word = 0, zero = 0;
    if (cudaMemcpy(&word, info.status_word, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(info.status_word, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return JET_ERR_CUDA;
    }
    if (detail) *detail = word;
    if (word == 0) return JET_OK;
    return (jet_status)(word & 0xFFu);
}

}  // extern "C"
