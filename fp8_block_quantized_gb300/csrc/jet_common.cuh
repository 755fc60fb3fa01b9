// Shared host/device helpers of the jet_fp8 library (sm_103a only).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "jet_fp8.h"

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

namespace jet {

// Facts about the current device, cached per device ordinal.
struct DeviceInfo {
    int ordinal;
    int num_sms;
    unsigned *status_word;  // device address of the library's status word
    void *context;          // the current CUDA context (a CUcontext), or null
};

// Checks that a current device exists and is sm_103; fills `info`.  Device
// addresses cached by the library are looked up again when the current
// context differs from the one they were looked up in (after a device reset
// the module, and its __device__ variables, may be loaded elsewhere).
jet_status current_device(DeviceInfo *info);

// The calling thread's current CUDA context (a CUcontext), or null.
void *current_context();

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline cudaStream_t as_stream(jet_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline jet_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? JET_OK : JET_ERR_CUDA;
}

// Launches a kernel of this library with programmatic dependent launch
// allowed: its blocks may start (barrier set-up, TMEM allocation) while the
// previous work on the stream is finishing.  Every such kernel calls
// griddep_wait() before it touches global memory, which waits until that
// previous work has completed and its writes are visible, so stream order is
// kept; the overlap hides the launch gap between short kernels.
template <typename... KArgs, typename... Args>
inline jet_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, args...) != cudaSuccess) {
        cudaGetLastError();
        return JET_ERR_CUDA;
    }
    return launch_status();
}

}  // namespace jet

// Early-return helpers for argument validation.
#define JET_REQUIRE(cond, code) \
    do {                        \
        if (!(cond)) return (code); \
    } while (0)

// ---------------------------------------------------------------------------
// Device side
// ---------------------------------------------------------------------------

namespace jet {

// Status word layout: low byte = jet_status code, bits 8..31 = wait site.
enum WaitSite : unsigned {
    SITE_GEMM_PRODUCER_EMPTY = 1,
    SITE_GEMM_MMA_FULL = 2,
    SITE_GEMM_MMA_TMEM_EMPTY = 3,
    SITE_GEMM_EPI_TMEM_FULL = 4,
    SITE_GEMM_DRAIN = 5,
    SITE_QUANT_STAGE = 6,
    SITE_TEST_NEVER_SET = 99,
};

__device__ __forceinline__ void report_timeout(unsigned *status_word, unsigned site) {
    // First error wins; later ones are dropped.
    atomicCAS(status_word, 0u, (site << 8) | (unsigned)JET_ERR_TIMEOUT);
}

// Programmatic dependent launch (see launch_pdl): allow the next kernel on
// the stream to start its blocks, and wait for the previous kernel's
// completion before touching global memory.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits longer than this many SM cycles (~2 s at 2 GHz) are treated as a
// hang: the waiting role records a timeout and abandons its work.  Healthy
// waits in these kernels last microseconds; the limit is far above them.
constexpr uint64_t kWaitLimitCycles = 4000000000ull;

}  // namespace jet
