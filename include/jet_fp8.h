/*
 * jet_fp8.h - C ABI of the GB300 (sm_103a) unified-precision FP8 linear layer.
 *
 * The layer is the one Jet-RL runs for both rollout and training ("Jet-RL:
 * Enabling On-Policy FP8 Reinforcement Learning with Unified Training and
 * Rollout Precision Flow", gist.science summary, sections "Kernarchitektur"
 * and "Quantisierungsschema"): activations and output gradients quantized to
 * E4M3 in 1x128 groups, weights in 128x128 blocks, each group with an FP32
 * scale ("NVIDIA强化学习加速实操：10分钟提升2倍训练效率", nmedialink.com,
 * section "为什么FP8适配线性层？", quantization table); forward, DGrad and WGrad
 * GEMMs in FP8, WGrad fed by 1x128 and 128x1 groups.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    allocates and frees nothing and keeps no pointer after a call returns.
 *  - Tensors are dense and row-major (last index contiguous).  BF16 values are
 *    passed as their uint16_t bit patterns; E4M3 codes as uint8_t (OCP E4M3FN:
 *    bias 7, max 448, NaN 0x7F/0xFF).  Scales are IEEE binary32.
 *  - Naming follows nn.Linear: X [M,K] (M tokens, K in-features), W [N,K]
 *    (N out-features), Y = X W^T [M,N], dY [M,N], dX = dY W [M,K],
 *    dW = dY^T X [N,K].  Kb = K/128, Nb = N/128, Mb = M/128.
 *  - The quantization rule for every group G: amax = max |v| over G (binary32),
 *    s = amax / 448 (IEEE binary32 division; s = 1 when amax == 0), and each
 *    code q = E4M3(fl32(v / s)) rounded to nearest, ties to even, saturating
 *    at +-448, sign of zero kept.  The stored scale dequantizes: v ~ q * s.
 *  - Every call validates its arguments on the host, in this order, and returns
 *    the first violation without launching anything: JET_ERR_NULL,
 *    JET_ERR_SHAPE, JET_ERR_ALIGN (every pointer must be 16-byte aligned),
 *    JET_ERR_WORKSPACE, JET_ERR_DEVICE (current device must be sm_103).
 *    A pointer may be NULL only when its tensor is empty.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  Launch failures return JET_ERR_CUDA.  Device-side
 *    bounded waits that give up are reported by jet_device_status().
 *  - Kernels are launched with programmatic dependent launch allowed: their
 *    blocks may start while earlier work on the stream finishes, but each
 *    waits for that work to complete before it reads or writes memory, so
 *    stream order holds (also inside captured CUDA graphs).
 *  - Non-finite inputs are outside the contract (their codes are unspecified).
 *  - Calls are reentrant; concurrent calls must not share output buffers.
 */
#ifndef JET_FP8_H
#define JET_FP8_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define JET_API __attribute__((visibility("default")))
#else
#define JET_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    JET_OK = 0,
    JET_ERR_NULL = 1,      /* a required pointer is NULL                       */
    JET_ERR_SHAPE = 2,     /* a size is negative or not a required multiple    */
    JET_ERR_ALIGN = 3,     /* a pointer is not 16-byte aligned                 */
    JET_ERR_CUDA = 4,      /* a CUDA runtime call or a kernel launch failed    */
    JET_ERR_DEVICE = 5,    /* no current device, or it is not sm_103           */
    JET_ERR_WORKSPACE = 6, /* workspace missing or smaller than required       */
    JET_ERR_TIMEOUT = 7    /* a device-side bounded wait gave up (see status)  */
} jet_status;

/* Operation ids for jet_workspace_bytes(). */
typedef enum {
    JET_OP_QUANT_ACT_1X128 = 0,
    JET_OP_QUANT_W_128X128 = 1,
    JET_OP_REQUANT_128X1 = 2,
    JET_OP_GEMM_FWD = 3,
    JET_OP_GEMM_DGRAD = 4,
    JET_OP_GEMM_WGRAD = 5,
    JET_OP_TOKEN_MULT_PROB_ERROR = 6,
    JET_OP_QUANT_DUAL_1X128_128X1 = 7,
    JET_OP_TOKEN_MISMATCH_MASKED = 8,
    JET_OP_SWIGLU_QUANT_1X128 = 9,
    JET_OP_KV_CALIBRATE = 10,
    JET_OP_KV_CACHE_WRITE = 11,
    JET_OP_TOKEN_MISMATCH_PER_SEQUENCE = 12,
    JET_OP_RMSNORM_QUANT_1X128 = 13
} jet_op;

/* A cudaStream_t handle passed as an opaque pointer. */
typedef void *jet_stream_t;

/* Static, NUL-terminated name of a status code ("JET_OK", ...). */
JET_API const char *jet_status_str(int status);

/* ABI version (major * 10000 + minor * 100 + patch). */
JET_API int jet_version(void);

/*
 * 1x128 quantization of activations or output gradients.
 * Source: nmedialink.com page, section "为什么FP8适配线性层？" (input activations
 * and output gradients: E4M3, [1,128], FP32 scales); gist.science summary,
 * "Quantisierungsschema" (activations 1x128).  Used for X before the forward
 * GEMM and for dY (with K := N) before the DGrad GEMM.
 *   x  [M][K] BF16 bits (in).       M >= 0, K >= 0 and K % 128 == 0.
 *   q  [M][K] E4M3 codes (out).
 *   s  [Kb][M] FP32 scales (out): s[kb*M + m] belongs to row m, columns
 *      128*kb .. 128*kb+127 (K-block-major so a GEMM tile's row scales are
 *      contiguous).
 */
JET_API jet_status jet_quant_act_1x128(const uint16_t *x, int64_t M, int64_t K,
                               uint8_t *q, float *s, jet_stream_t stream);

/*
 * 128x128 block quantization of weights (run once per weight sync).
 * Source: nmedialink.com page, quantization table (weights: E4M3, [128,128],
 * FP32); gist.science summary, "Quantisierungsschema" (weights 128x128).
 *   w  [N][K] BF16 bits (in).       N, K >= 0, both multiples of 128.
 *   q  [N][K] E4M3 codes (out).
 *   s  [Nb][Kb] FP32 scales (out), s[nb*Kb + kb].
 */
JET_API jet_status jet_quant_w_128x128(const uint16_t *w, int64_t N, int64_t K,
                               uint8_t *q, float *s, jet_stream_t stream);

/*
 * 128x1 re-quantization along the token axis, fused with the transpose that
 * the WGrad GEMM needs.  Source: 163.com article, section 五 (1x128 forward
 * groups re-quantized as 128x1 in backward); gist.science summary,
 * "Quantisierungsschema" (WGrad with 1x128 and 128x1 groups).  The input is
 * the saved FP8 form: v[m][k] = fl32(D4(q[m][k]) * s[k/128][m]); each group is
 * tokens 128*mb .. 128*mb+127 of one column k.
 *   q   [M][K] E4M3 codes, s [Kb][M] scales (in; the jet_quant_act_1x128 form).
 *   qT  [K][M] E4M3 codes (out), transposed.   M, K >= 0, multiples of 128.
 *   sT  [Mb][K] FP32 scales (out), sT[mb*K + k].
 */
JET_API jet_status jet_requant_128x1(const uint8_t *q, const float *s, int64_t M,
                             int64_t K, uint8_t *qT, float *sT,
                             jet_stream_t stream);

/*
 * SwiGLU with the 1x128 quantization of its output fused: the input of an
 * MLP's down projection, h = silu(gate) * up, written directly as the
 * jet_quant_act_1x128 form (no BF16 copy of h).  Source: 163.com article,
 * section 三, and gist.science summary, "Quantisierungsschema" (the quantizer
 * fused into the operator that produces a linear layer's input).  h is
 * evaluated in binary32 by a fixed sequence of IEEE operations (Cody-Waite
 * e^x with a degree-7 Taylor polynomial; 1/(1 + e^-g) by a bit-pattern seed
 * and three Newton-Raphson steps; g < -80 gives a signed zero), within 3 ulps
 * of silu(g) * up; its 128-wide groups then follow the 1x128 group rule.
 *   gate, up  BF16 bits, row m at gate + m*ld and up + m*ld (in).  For the
 *       concatenated [M][2F] output of a gate_up product pass gate = base,
 *       up = base + F, ld = 2F.  ld >= F, a multiple of 8.
 *   q   [M][F] E4M3 codes, s [F/128][M] FP32 scales (out).  M, F >= 0, F a
 *       multiple of 128.  Non-finite h (overflowing products) is a
 *       precondition violation with unspecified codes.
 */
JET_API jet_status jet_swiglu_quant_1x128(const uint16_t *gate, const uint16_t *up, int64_t ld,
                                          int64_t M, int64_t F, uint8_t *q, float *s,
                                          jet_stream_t stream);

/*
 * RMSNorm with the 1x128 quantization of its output fused: the input of the
 * q/k/v and gate/up projections written as E4M3 codes and FP32 scales
 * straight from the residual stream, with no BF16 normalised activation.
 * Source: gist.science summary, "Implementierung" (fused activation/RMSNorm
 * operators in custom kernels), and 163.com article, section 五 (a linear
 * layer's input quantized in the operator that produces it).  The pages give
 * no arithmetic; y = x * g / sqrt(mean(x^2) + eps) is evaluated in binary32
 * in one fixed order: lane partial sums of squares (lane l adds the elements
 * 8 (32 j + l) + t in order of j, then t = 0 .. 7), a five-level butterfly,
 * ms = ss / K, v = ms + eps, r = 1 / sqrt(v) (IEEE operations; r = 0 when
 * v == 0), y = (x * r) * g; its 128-wide groups then follow the 1x128 group
 * rule.  Within a few ulps of binary64 RMSNorm (at most (K/64 + 8.5) 2^-24
 * relative).
 *   x   [M][K] BF16 bits (in; the residual stream), g [K] BF16 bits (in; the
 *       norm's gain).  M, K >= 0, K a multiple of 128 and below 2^24.
 *   eps >= 0 (finite); the model's value, e.g. 1e-5.
 *   q   [M][K] E4M3 codes, s [K/128][M] FP32 scales (out).
 * Rows whose sum of squares overflows binary32 are a precondition violation
 * with unspecified codes.
 */
JET_API jet_status jet_rmsnorm_quant_1x128(const uint16_t *x, const uint16_t *g, int64_t M,
                                           int64_t K, float eps, uint8_t *q, float *s,
                                           jet_stream_t stream);

/*
 * FP8 KV cache, scales recalibrated after each model update.  Source: FP8-RL
 * article (m.66260.cn), KV-cache paragraph (scale factors calibrated again
 * after every model update); nmedialink page, section "FP8探索新维度：KV缓存与
 * 注意力机制赋能" (FP8 KV cache).  The pages give no granularity; here one
 * FP32 scale per KV head, for K and for V separately.
 *
 * jet_kv_calibrate: scale[h] = amax_h / 448 (IEEE division; 1 when the head
 * is all zero), amax_h over all T tokens and D channels of head h of the
 * calibration batch x [T][H][D] (BF16 bits).  Writes scale [H] FP32 (device;
 * also used as scratch during the call).
 *
 * jet_kv_cache_write: cache[slots[t]][h][d] = E4(fl32(x[t][h][d] / scale[h]))
 * for the T new entries x [T][H][D] (BF16 bits); entries beyond the
 * calibrated range saturate to +-448.  slots [T] int64 DEVICE array of
 * distinct cache rows; a slot outside [0, S) is skipped.  cache [S][H][D]
 * E4M3 codes (in/out; other rows untouched).
 *
 * T, S >= 0; 0 <= H <= 1024; D a multiple of 16.
 */
JET_API jet_status jet_kv_calibrate(const uint16_t *x, int64_t T, int64_t H, int64_t D,
                                    float *scale, jet_stream_t stream);
JET_API jet_status jet_kv_cache_write(const uint16_t *x, const float *scale,
                                      const int64_t *slots, int64_t T, int64_t H, int64_t D,
                                      uint8_t *cache, int64_t S, jet_stream_t stream);

/*
 * Both quantizations of one tensor from a single read: the 1x128 form of
 * jet_quant_act_1x128 and the transposed 128x1 form that jet_requant_128x1
 * derives from it (re-quantized from the FP8 1x128 values).  Used for the
 * output gradient dY, whose two forms feed DGrad and WGrad in the same
 * backward step.  Source: 163.com article, section 五 (1x128 groups
 * re-quantized as 128x1 for backward; quantization fused into the operator
 * that produces the tensor); gist.science summary, "Quantisierungsschema"
 * (DGrad with 1x128, WGrad with 1x128 and 128x1).  Codes and scales equal
 * those of jet_quant_act_1x128 followed by jet_requant_128x1, bit for bit.
 *   x   [M][K] BF16 bits (in).      M, K >= 0, both multiples of 128.
 *   q   [M][K] E4M3 codes, s [Kb][M] FP32 scales (out; the 1x128 form).
 *   qT  [K][M] E4M3 codes, sT [Mb][K] FP32 scales (out; the 128x1 form).
 */
JET_API jet_status jet_quant_dual_1x128_128x1(const uint16_t *x, int64_t M, int64_t K,
                                              uint8_t *q, float *s, uint8_t *qT, float *sT,
                                              jet_stream_t stream);

/*
 * Forward GEMM  Y = X W^T  with per-128-K-block scale promotion:
 *   Y[m][n] = sum_kb sx[kb][m] * sw[n/128][kb] * sum_{k in kb} qx[m][k] qw[n][k]
 * accumulated in FP32 and written as BF16 (round to nearest even).
 * Source: gist.science summary, "Quantisierungsschema" (FP8 GEMMs of linear
 * layers); 163.com article, section 五 (1x128 inputs times 128x128 weights).
 *   qx [M][K], sx [Kb][M] (jet_quant_act_1x128 of X);  M >= 0.
 *   qw [N][K], sw [Nb][Kb] (jet_quant_w_128x128 of W); N, K multiples of 128.
 *   y  [M][N] BF16 bits (out).  K == 0 writes zeros.
 *   ws / ws_bytes: device workspace of at least
 *   jet_workspace_bytes(JET_OP_GEMM_FWD, M, N, K) bytes, else JET_ERR_WORKSPACE
 *   (NULL/0 allowed when that is 0).  It can be non-zero only for M <= 512,
 *   where the contraction may be split into ranges whose FP32 partial tiles
 *   [splits][M][N] go to ws and are then summed in a fixed order and rounded
 *   once to BF16; the split depends only on (M, N, K), so results are the same
 *   on every call and every device.  Its contents need no initialisation and
 *   are scratch after the call; concurrent calls need separate workspaces.
 *   M == 1, and 2 <= M <= 4 with M * N * K <= 2^25 (decode), run a weight-streaming kernel
 *   on CUDA cores with the same arithmetic (exact code products, FP32 sums
 *   per scale group, scaled and summed in a fixed order) and needs no
 *   workspace.
 */
JET_API jet_status jet_gemm_fp8_fwd(const uint8_t *qx, const float *sx,
                            const uint8_t *qw, const float *sw, int64_t M,
                            int64_t N, int64_t K, uint16_t *y, void *ws,
                            size_t ws_bytes, jet_stream_t stream);

/*
 * Grouped forward GEMM of expert linears (mixture-of-experts layers), one
 * launch for all experts:  for every expert e and its tokens
 * m in [offsets[e], offsets[e+1]),
 *   Y[m][n] = sum_kb sx[kb][m] * sw[e][n/128][kb] * sum_{k in kb} qx[m][k] qw[e][n][k]
 * with the arithmetic of jet_gemm_fp8_fwd (FP32 accumulation, BF16 out).
 * Source: 163.com article / nmedialink.com page (FP8 for the Qwen3-30B MoE
 * model, section "在专家混合模型中的突破"); m.66260.cn FP8-RL article (expert
 * layers in the compressed format).  The pages give no grouped kernel; this
 * layout is this library's choice.
 *   qx [M][K], sx [Kb][M]: the tokens of all experts, in expert order (the
 *     jet_quant_act_1x128 form of the concatenated activations).
 *   qw [E][N][K], sw [E][Nb][Kb]: the experts' weights and scales, stacked.
 *   offsets [E+1] int64, DEVICE array: offsets[0] = 0, non-decreasing,
 *     offsets[E] = M (e.g. written by the routing kernel).  Offsets outside
 *     [0, M] are clamped and a decreasing pair is an empty expert, so no
 *     write ever leaves y; results are then unspecified.
 *   y [M][N] BF16 bits (out).  1 <= E <= 384; N, K multiples of 128.
 */
JET_API jet_status jet_gemm_fp8_fwd_grouped(const uint8_t *qx, const float *sx,
                                            const uint8_t *qw, const float *sw,
                                            const int64_t *offsets, int64_t E, int64_t M,
                                            int64_t N, int64_t K, uint16_t *y,
                                            jet_stream_t stream);

/*
 * Grouped DGrad of expert linears, one launch: for every expert e and its
 * tokens m in [offsets[e], offsets[e+1]),
 *   dX[m][k] = sum_nb sdy[nb][m] * sw[e][nb][k/128] * sum_{n in nb} qdy[m][n] qw[e][n][k]
 * with the arithmetic of jet_gemm_fp8_dgrad.  Source and layout as
 * jet_gemm_fp8_fwd_grouped (the backward of the same expert linears).
 *   qdy [M][N], sdy [Nb][M]: the output gradients of all experts' tokens in
 *     expert order.  qw [E][N][K], sw [E][Nb][Kb] as in the forward.
 *   offsets [E+1] int64 DEVICE array, as in jet_gemm_fp8_fwd_grouped.
 *   dx [M][K] BF16 bits (out).  1 <= E <= 384; N, K multiples of 128.
 */
JET_API jet_status jet_gemm_fp8_dgrad_grouped(const uint8_t *qdy, const float *sdy,
                                              const uint8_t *qw, const float *sw,
                                              const int64_t *offsets, int64_t E, int64_t M,
                                              int64_t N, int64_t K, uint16_t *dx,
                                              jet_stream_t stream);

/*
 * Grouped WGrad of expert linears, one launch: every expert's weight
 * gradient over its own tokens,
 *   dW[e][n][k] = sum_{mb in expert e} sdyT[mb][n] * sxT[mb][k]
 *                 * sum_{m in mb} qdyT[n][m] qxT[k][m]
 * with the arithmetic of jet_gemm_fp8_wgrad.  Source as
 * jet_gemm_fp8_fwd_grouped; 128x1 groups as jet_gemm_fp8_wgrad.
 *   qdyT [N][M], sdyT [Mb][N] and qxT [K][M], sxT [Mb][K]: the 128x1 forms
 *     (jet_requant_128x1 / jet_quant_dual_1x128_128x1) of the expert-ordered
 *     output gradients and inputs.
 *   offsets [E+1] int64 DEVICE array: offsets[0] = 0, non-decreasing,
 *     offsets[E] = M, every offset a multiple of 128 (a 128-token group never
 *     straddles two experts: experts are padded to whole groups, with zero
 *     rows).  Offsets are clamped to [0, M]; other violations give
 *     unspecified results, never a write outside dw.
 *   dw [E][N][K] BF16 bits (out); an expert without tokens gets zeros.
 *   M, N, K multiples of 128; 1 <= E <= 384.
 */
JET_API jet_status jet_gemm_fp8_wgrad_grouped(const uint8_t *qdyT, const float *sdyT,
                                              const uint8_t *qxT, const float *sxT,
                                              const int64_t *offsets, int64_t E, int64_t M,
                                              int64_t N, int64_t K, uint16_t *dw,
                                              jet_stream_t stream);

/*
 * DGrad GEMM  dX = dY W :
 *   dX[m][k] = sum_nb sdy[nb][m] * sw[nb][k/128] * sum_{n in nb} qdy[m][n] qw[n][k]
 * FP32 accumulation, BF16 out.  Source: gist.science summary,
 * "Quantisierungsschema", "Backward-Pass" (DGrad in FP8).
 *   qdy [M][N], sdy [Nb][M] (jet_quant_act_1x128 of dY with K := N).
 *   qw  [N][K], sw [Nb][Kb] (the forward weight codes, read transposed).
 *   dx  [M][K] BF16 bits (out).  N == 0 writes zeros.
 *   ws / ws_bytes: as for the forward GEMM, with
 *   jet_workspace_bytes(JET_OP_GEMM_DGRAD, M, N, K) (partials [splits][M][K]).
 */
JET_API jet_status jet_gemm_fp8_dgrad(const uint8_t *qdy, const float *sdy,
                              const uint8_t *qw, const float *sw, int64_t M,
                              int64_t N, int64_t K, uint16_t *dx, void *ws,
                              size_t ws_bytes, jet_stream_t stream);

/*
 * WGrad GEMM  dW = dY^T X  on the 128x1 (token-axis) groups:
 *   dW[n][k] = sum_mb sdyT[mb][n] * sxT[mb][k] * sum_{m in mb} qdyT[n][m] qxT[k][m]
 * FP32 accumulation, BF16 out.  Source: gist.science summary,
 * "Quantisierungsschema", "Backward-Pass" (WGrad in FP8 with 1x128 and 128x1).
 *   qdyT [N][M], sdyT [Mb][N]  (jet_requant_128x1 of dY's 1x128 form).
 *   qxT  [K][M], sxT  [Mb][K]  (jet_requant_128x1 of X's 1x128 form).
 *   dw   [N][K] BF16 bits (out).  M % 128 == 0; M == 0 writes zeros.
 *   ws / ws_bytes: unused (jet_workspace_bytes(JET_OP_GEMM_WGRAD, ...) is 0).
 */
JET_API jet_status jet_gemm_fp8_wgrad(const uint8_t *qdyT, const float *sdyT,
                              const uint8_t *qxT, const float *sxT, int64_t M,
                              int64_t N, int64_t K, uint16_t *dw, void *ws,
                              size_t ws_bytes, jet_stream_t stream);

/*
 * Train/rollout mismatch metric
 *   token-mult-prob-error = (1/n) * sum_i exp(|logp_train[i] - logp_rollout[i]|)
 * Source: nmedialink.com page, section "FP8面临的关键挑战：数值分歧".  No mask:
 * every one of the n tokens counts.  Per-thread sums in FP32, across threads
 * and blocks in FP64 (fixed order, deterministic); result written as FP32.
 *   logp_train, logp_rollout [n] FP32 (in), n >= 1.
 *   out: one FP32 in device memory (out).
 *   ws / ws_bytes: at least jet_workspace_bytes(JET_OP_TOKEN_MULT_PROB_ERROR,
 *   n, 0, 0) bytes of device memory (per-block FP64 partial sums).
 */
JET_API jet_status jet_token_mult_prob_error(const float *logp_train,
                                     const float *logp_rollout, int64_t n,
                                     float *out, void *ws, size_t ws_bytes,
                                     jet_stream_t stream);

/*
 * token-mult-prob-error without a workspace argument, for callers that cannot
 * allocate device memory: a plain C host that only receives device pointers
 * from another runtime and has no allocator of its own, or a latency-bound
 * loop that must not call cudaMalloc (it can synchronize the whole device and
 * is not ordered on a stream).  The pages have no counterpart; this is a
 * convenience of this library.  Same arithmetic, grid and result as
 * jet_token_mult_prob_error.
 *   logp_train, logp_rollout [n] FP32 (in), out: one FP32 (out); device
 *   pointers owned by the caller, as everywhere else.
 *   1 <= n <= 2,097,152; larger n returns JET_ERR_SHAPE before any launch.
 * The per-block partial sums go to a static 8 KB device array inside the
 * library (1024 FP64 slots; every device that loads the library keeps it until
 * the process exits).  The library allocates and frees nothing here.  The first
 * call on a device looks up that array's device address (with the device
 * current) and caches it for the device's current context (after a device
 * reset the next call looks it up again); make that first call before any
 * stream capture.
 * All calls share the one array: calls whose kernels overlap on the GPU (e.g.
 * on two streams at once) race on it and may return wrong values - order them
 * on one stream or use jet_token_mult_prob_error with separate workspaces.
 * Nothing needs clearing between calls: every slot a call reads is written
 * earlier in the same call.
 */
JET_API jet_status jet_token_mult_prob_error_noalloc(const float *logp_train,
                                                     const float *logp_rollout,
                                                     int64_t n, float *out,
                                                     jet_stream_t stream);

/*
 * The mismatch metric over a subset of the tokens, fused with the per-token
 * importance weights of the training loss, in one pass over the tokens.
 * Source: nmedialink.com page, sections "FP8面临的关键挑战：数值分歧" (the
 * metric) and "重要抽样技术：提升RL精度的尖兵" (importance sampling with FP8);
 * m.66260.cn FP8-RL article (the weight is the ratio of the original to the
 * compressed model's token probability).  With a = logp_train, b =
 * logp_rollout and mask m (the tokens that count, e.g. a response mask):
 *   w_i = m_i ? min(exp(a_i - b_i), cap) : 0        (no cap when cap <= 0;
 *                                                    the pages give none)
 *   out = sum_{m_i} exp(|a_i - b_i|) / count,  count = #{i : m_i != 0}
 * exp in FP32 per token, sums in FP32 per thread and FP64 across threads and
 * blocks in a fixed order; out is NaN when no token counts.
 *   logp_train, logp_rollout [n] FP32 (in), n >= 1.
 *   mask [n] uint8 (in; nonzero = the token counts), or NULL: every token.
 *   w [n] FP32 (out), or NULL: the weights are not written.
 *   out: one FP32 (out); count: one int64 (out), or NULL.  Device pointers.
 *   ws / ws_bytes: at least jet_workspace_bytes(JET_OP_TOKEN_MISMATCH_MASKED,
 *   n, 0, 0) bytes of device memory.
 */
JET_API jet_status jet_token_mismatch_masked(const float *logp_train, const float *logp_rollout,
                                             const uint8_t *mask, int64_t n, float cap, float *w,
                                             float *out, int64_t *count, void *ws,
                                             size_t ws_bytes, jet_stream_t stream);

/*
 * Per-sequence form of jet_token_mismatch_masked, one pass: for every
 * sequence s (tokens seq_offsets[s] .. seq_offsets[s+1]) the mean of
 * exp|logp_train_i - logp_rollout_i| over its masked tokens, and the same
 * per-token importance weights.  Source: nmedialink page, "FP8面临的关键挑战：
 * 数值分歧" (the metric) and its importance-sampling paragraph; FP8-RL article
 * (the probability ratio).  Computed as jet_token_mismatch_masked: exp in
 * FP32 per token, sums in FP64, result FP32; deterministic.
 *   logp_train, logp_rollout [n] FP32; mask [n] uint8 or NULL (every token).
 *   seq_offsets [S+1] int64 DEVICE array: 0, non-decreasing, n (offsets are
 *     clamped to [0, n]; a decreasing pair is an empty sequence).
 *   cap: importance weights min(w, cap) when cap > 0.
 *   w [n] FP32 or NULL (out); out [S] FP32 (out; NaN for a sequence without
 *   masked tokens); count [S] int64 or NULL (out).  S >= 1, n >= 0.
 */
JET_API jet_status jet_token_mismatch_per_sequence(const float *logp_train,
                                                   const float *logp_rollout,
                                                   const uint8_t *mask,
                                                   const int64_t *seq_offsets, int64_t S,
                                                   int64_t n, float cap, float *w, float *out,
                                                   int64_t *count, jet_stream_t stream);

/*
 * Workspace bytes an operation needs for the given sizes (0 if none).
 * For JET_OP_TOKEN_MULT_PROB_ERROR and JET_OP_TOKEN_MISMATCH_MASKED pass n as M.  Returns 0 for negative sizes
 * or an unknown op.  Pure host function; needs no device.
 */
JET_API size_t jet_workspace_bytes(int op, int64_t M, int64_t N, int64_t K);

/*
 * Synchronizes `stream`, then reads and clears the device-side status word of
 * the current device.  Returns JET_OK, JET_ERR_TIMEOUT (a bounded wait inside
 * a kernel gave up; the kernel skipped its remaining work and released its
 * resources, so the context stays usable) or JET_ERR_CUDA (the synchronize
 * itself failed).  If `detail` is not NULL it receives the raw status word
 * (0 when clean; otherwise the code in the low byte and the wait site above).
 */
JET_API jet_status jet_device_status(jet_stream_t stream, uint32_t *detail);

/*
 * Self-test of the failure path every pipelined kernel uses: launches one
 * block that waits on a barrier nothing completes, with a limit of
 * `limit_us` microseconds at the maximum SM clock (1 .. 1,000,000; the wait
 * is counted in SM cycles, so it lasts longer at lower clocks).  The wait gives up, records
 * JET_ERR_TIMEOUT in the device status word and the kernel returns, so a
 * following jet_device_status() reports JET_ERR_TIMEOUT and the context stays
 * usable.  The pages have no counterpart; it exists to test the bounded waits.
 */
JET_API jet_status jet_selftest_bounded_wait(uint32_t limit_us, jet_stream_t stream);

/*
 * Self-test of the GEMM's own failure path: runs the forward product
 * Y = X W^T (same operands and layouts as jet_gemm_fp8_fwd, M <= 128 tokens,
 * on the single-CTA tensor-core kernel, contraction not split) with every
 * pipeline wait limited to `limit_cycles` SM cycles (1 .. 4e9; the library's
 * GEMMs use 4e9, about 2 s).  With a limit shorter than the first operand
 * load, a role of the kernel gives up: it records JET_ERR_TIMEOUT and its wait
 * site (1 producer, 2 MMA issuer waiting for operands, 3 MMA issuer waiting
 * for an accumulator, 4 promotion warps) in the device status word and sets
 * the CTA's abort flag; the other roles stop at their next wait, the producer
 * waits for its loads in flight, the MMA issuer for its MMAs, TMEM is freed
 * and the kernel returns, so jet_device_status() reports JET_ERR_TIMEOUT and
 * the context stays usable.  Y is then unspecified.  Same argument checks as
 * jet_gemm_fp8_fwd, plus M <= 128 and the limit's range (JET_ERR_SHAPE).
 * The pages have no counterpart; it exists to test the bounded waits.
 */
JET_API jet_status jet_selftest_gemm_timeout(const uint8_t *qx, const float *sx,
                                             const uint8_t *qw, const float *sw, int64_t M,
                                             int64_t N, int64_t K, uint16_t *y,
                                             uint64_t limit_cycles, jet_stream_t stream);

/*
 * Self-test of the division the quantizers use: q[i] = x[i] / s[i] computed
 * exactly as a quantizer divides a value x by its group scale s (a
 * reciprocal of s shared by the group and Markstein's correction steps).  It
 * equals the IEEE binary32 quotient whenever s >= 2^-90 and |x/s| >= 2^-11,
 * and for every pair when s < 2^-90; smaller quotients agree in sign and lie
 * below 2^-10, so their E4M3 codes are the same.  x, s, q: [n] FP32 device
 * arrays.  The pages have no counterpart; it exists to test that division.
 */
JET_API jet_status jet_selftest_quotient(const float *x, const float *s, int64_t n, float *q,
                                         jet_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* JET_FP8_H */
