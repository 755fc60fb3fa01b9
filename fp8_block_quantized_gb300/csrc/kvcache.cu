// FP8 KV cache with the scale factors recalibrated after every model update
// ("FP8-RL" article (m.66260.cn), the KV-cache paragraph; nmedialink page,
// "FP8探索新维度：KV缓存与注意力机制赋能").  One binary32 scale per KV head (K
// and V each): s_h = amax_h / 448 over the calibration tokens, 1 when the
// head is all zero (the group rule's scale, quant_rule.cuh); every entry
// written afterwards is E4(fl32(x / s_h)), saturating beyond the calibrated
// range.
//
// Calibration: the scale array is zeroed, one pass over the tokens takes each
// head's amax (16-byte loads, per-thread or per-CTA maxima, one global
// atomicMax per head and CTA on the amax's bit pattern, which orders like
// the value for non-negative floats, so the result does not depend on the
// order), and a one-block pass turns the amaxes into scales in place.
// Cache write: each thread takes 8 consecutive channels of a new entry (one
// 16-byte load, one 8-byte store into the entry's slot), dividing by the
// head's scale with the group rule's correctly rounded division.  Both are
// bound by HBM.
#include "jet_common.cuh"
#include "stream_ld.cuh"
#include "quant_rule.cuh"

namespace {

constexpr int kKvThreads = 256;
constexpr int kKvCtasPerSm = 4;
constexpr int64_t kKvMaxHeads = 1024;

// max(|x|) of eight BF16 values, as a bit pattern (non-negative float)
__device__ __forceinline__ uint32_t amax8_bits(const uint4 &v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = (w[i] << 16) & 0x7FFFFFFFu, hi = w[i] & 0x7FFF0000u;
        m = max(m, max(lo, hi));
    }
    return m;
}

// Both kernels walk the 8-channel chunks c of x[T][H][D] (row8 = H D / 8
// chunks per token) with a grid stride.  When the stride is a multiple of
// row8 (the host picks such a grid whenever row8 divides or is a multiple of
// the block size), a thread's chunks all sit at the same place j of their
// tokens, hence in the same head: its head, divisor and running maximum stay
// in registers and the token advances by stride / row8 without a division.
// Otherwise each chunk finds its token and head by division.  kUnroll chunks
// are loaded before any of them is used.
constexpr int kUnroll = 4;

// amax[h] (bit patterns, zeroed by the caller) over x[T][H][D].
template <bool kFixed>
__global__ void __launch_bounds__(kKvThreads)
kv_amax_kernel(const uint16_t *__restrict__ x, int64_t T, int H, int D,
               unsigned *__restrict__ amax) {
    extern __shared__ unsigned head_max[];
    for (int h = threadIdx.x; h < H; h += blockDim.x) head_max[h] = 0u;
    __syncthreads();
    const int64_t row8 = (int64_t)H * D / 8;  // 8-channel chunks per token
    const int64_t n = T * row8;
    const int d8 = D / 8;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t c = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    uint32_t mine = 0;  // kFixed: this thread's head maximum
    for (; c < n; c += kUnroll * stride) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (c + u * stride < n) v[u] = ld_stream16(x + 8 * (c + u * stride));
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (c + u * stride >= n) break;
            const uint32_t m = amax8_bits(v[u]);
            if constexpr (kFixed) {
                mine = max(mine, m);
            } else if (m) {
                atomicMax(&head_max[(int)(((c + u * stride) % row8) / d8)], m);
            }
        }
    }
    if constexpr (kFixed) {
        const int64_t c0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
        if (mine) atomicMax(&head_max[(int)((c0 % row8) / d8)], mine);
    }
    __syncthreads();
    for (int h = threadIdx.x; h < H; h += blockDim.x)
        if (head_max[h]) atomicMax(&amax[h], head_max[h]);
}

// scale[h] = amax_h / 448 (1 if amax_h = 0), in place over the amax bits.
__global__ void __launch_bounds__(kKvThreads) kv_scale_kernel(float *scale, int H) {
    jet::griddep_launch_dependents();
    jet::griddep_wait();
    for (int h = threadIdx.x; h < H; h += blockDim.x)
        scale[h] = group_scale(__uint_as_float(reinterpret_cast<unsigned *>(scale)[h]));
}

__device__ __forceinline__ uint2 encode8(const uint4 &v, const Divisor &dv) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float nf[8];  // -x, for the division routine
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        nf[2 * i] = __uint_as_float((w[i] << 16) ^ 0x80000000u);
        nf[2 * i + 1] = __uint_as_float((w[i] & 0xFFFF0000u) ^ 0x80000000u);
    }
    uint2 out;
    out.x = encode4(nf, dv);
    out.y = encode4(nf + 4, dv);
    return out;
}

template <bool kFixed>
__global__ void __launch_bounds__(kKvThreads, kKvCtasPerSm)
kv_write_kernel(const uint16_t *__restrict__ x, const float *__restrict__ scale,
                const int64_t *__restrict__ slot, int64_t T, int H, int D,
                uint8_t *__restrict__ cache, int64_t S) {
    extern __shared__ float2 head_div[];  // (s, -RN(1/s)), general path only
    jet::griddep_launch_dependents();
    jet::griddep_wait();
    const int64_t row8 = (int64_t)H * D / 8;
    const int64_t n = T * row8;
    const int d8 = D / 8;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t c0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if constexpr (kFixed) {
        const int64_t j = c0 % row8, dt = stride / row8;
        const Divisor dv = make_divisor(scale[j / d8]);
        for (int64_t t = c0 / row8; t < T; t += kUnroll * dt) {
            uint4 v[kUnroll];
            int64_t sl[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t tu = t + u * dt;
                sl[u] = tu < T ? slot[tu] : -1;
                if (tu < T) v[u] = ld_stream16(x + 8 * (tu * row8 + j));
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (sl[u] >= 0 && sl[u] < S)
                    *reinterpret_cast<uint2 *>(cache + (sl[u] * row8 + j) * 8) = encode8(v[u], dv);
        }
    } else {
        for (int h = threadIdx.x; h < H; h += blockDim.x) {
            const Divisor dv = make_divisor(scale[h]);
            head_div[h] = make_float2(dv.s, dv.ny);
        }
        __syncthreads();
        for (int64_t c = c0; c < n; c += stride) {
            const int64_t t = c / row8, j = c - t * row8;
            const int64_t sl = slot[t];
            if (sl < 0 || sl >= S) continue;
            const float2 hd = head_div[j / d8];
            Divisor dv;
            dv.s = hd.x;
            dv.ny = hd.y;
            dv.fast = hd.x >= 0x1p-90f;
            *reinterpret_cast<uint2 *>(cache + (sl * row8 + j) * 8) =
                encode8(ld_stream16(x + 8 * c), dv);
        }
    }
}

// A grid whose thread count is a multiple of row8 when one exists near the
// wanted size (then kFixed); else the wanted size.
int64_t kv_grid(int64_t want, int64_t cap, int64_t row8, bool *fixed) {
    int64_t g = want < cap ? want : cap;
    if (g < 1) g = 1;
    *fixed = false;
    if (kKvThreads % row8 == 0) {
        *fixed = true;
    } else if (row8 % kKvThreads == 0) {
        const int64_t m = row8 / kKvThreads;  // CTAs per token row
        if (m <= cap) {
            g = (g + m - 1) / m * m;
            if (g > cap) g = cap / m * m;
            *fixed = true;
        }
    }
    return g;
}

jet_status check_kv(int64_t T, int64_t H, int64_t D) {
    if (T < 0 || H < 0 || D < 0) return JET_ERR_SHAPE;
    if (H > kKvMaxHeads || D % 16 != 0 || T >= ((int64_t)1 << 40) || H * D >= ((int64_t)1 << 30))
        return JET_ERR_SHAPE;
    return JET_OK;
}

}  // namespace

jet_status jet_kv_calibrate(const uint16_t *x, int64_t T, int64_t H, int64_t D, float *scale,
                            jet_stream_t stream) {
    jet_status st = check_kv(T, H, D);
    if (st != JET_OK) return st;
    JET_REQUIRE(H == 0 || scale, JET_ERR_NULL);
    JET_REQUIRE(T * H * D == 0 || x, JET_ERR_NULL);
    JET_REQUIRE(jet::aligned16(x) && jet::aligned16(scale), JET_ERR_ALIGN);
    jet::DeviceInfo dev;
    st = jet::current_device(&dev);
    if (st != JET_OK) return st;
    if (H == 0) return JET_OK;
    cudaStream_t s = jet::as_stream(stream);
    if (cudaMemsetAsync(scale, 0, (size_t)H * sizeof(float), s) != cudaSuccess) return JET_ERR_CUDA;
    const int64_t chunks = T * H * D / 8;
    if (chunks > 0) {
        const int64_t want = (chunks + kUnroll * kKvThreads - 1) / (kUnroll * kKvThreads);
        bool fixed;
        const int64_t g = kv_grid(want, (int64_t)dev.num_sms * kKvCtasPerSm, H * D / 8, &fixed);
        // a plain launch: it must follow the zeroing memset entirely
        auto *kernel = fixed ? kv_amax_kernel<true> : kv_amax_kernel<false>;
        kernel<<<dim3((unsigned)g), dim3(kKvThreads), (size_t)H * sizeof(unsigned), s>>>(
            x, T, (int)H, (int)D, reinterpret_cast<unsigned *>(scale));
        if (cudaGetLastError() != cudaSuccess) return JET_ERR_CUDA;
    }
    return jet::launch_pdl(kv_scale_kernel, dim3(1), dim3(kKvThreads), 0, s, scale, (int)H);
}

jet_status jet_kv_cache_write(const uint16_t *x, const float *scale, const int64_t *slots,
                              int64_t T, int64_t H, int64_t D, uint8_t *cache, int64_t S,
                              jet_stream_t stream) {
    jet_status st = check_kv(T, H, D);
    if (st != JET_OK) return st;
    JET_REQUIRE(S >= 0, JET_ERR_SHAPE);
    const bool empty = T == 0 || H == 0 || D == 0;
    JET_REQUIRE(empty || (x && scale && slots && cache), JET_ERR_NULL);
    JET_REQUIRE(jet::aligned16(x) && jet::aligned16(scale) && jet::aligned16(slots) &&
                    jet::aligned16(cache),
                JET_ERR_ALIGN);
    jet::DeviceInfo dev;
    st = jet::current_device(&dev);
    if (st != JET_OK) return st;
    if (empty) return JET_OK;
    const int64_t chunks = T * H * D / 8;
    const int64_t want = (chunks + kUnroll * kKvThreads - 1) / (kUnroll * kKvThreads);
    bool fixed;
    const int64_t g = kv_grid(want, (int64_t)dev.num_sms * kKvCtasPerSm, H * D / 8, &fixed);
    if (fixed)
        return jet::launch_pdl(kv_write_kernel<true>, dim3((unsigned)g), dim3(kKvThreads), 0,
                               jet::as_stream(stream), x, scale, slots, T, (int)H, (int)D, cache,
                               S);
    return jet::launch_pdl(kv_write_kernel<false>, dim3((unsigned)g), dim3(kKvThreads),
                           (size_t)H * sizeof(float2), jet::as_stream(stream), x, scale, slots, T,
                           (int)H, (int)D, cache, S);
}
