/*
 * Plain CPU oracle for the unified-precision FP8 linear layer (Jet-RL).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * statement of what the GPU path computes.  Only the test-suite, the smoke
 * check and the CPU-baseline leg of the benchmark may load it; the product
 * library never links, calls or falls back to it, and it shares no code,
 * header, table or constant generator with the CUDA sources.
 *
 * What each part follows:
 *   - Quantization granularities and scale type: "NVIDIA强化学习加速实操：10分钟
 *     提升2倍训练效率" (nmedialink.com), section "为什么FP8适配线性层？", the
 *     quantization table: weights E4M3 in [128,128] blocks, input activations
 *     and output gradients E4M3 in [1,128] groups, FP32 block scales.
 *   - Activations 1x128 / weights 128x128: "Jet-RL: Enabling On-Policy FP8
 *     Reinforcement Learning with Unified Training and Rollout Precision Flow"
 *     (gist.science), section "Quantisierungsschema".
 *   - Backward: DGrad and WGrad GEMMs in FP8, WGrad fed by 1x128 and 128x1
 *     groups: same page, same section, "Backward-Pass".
 *   - Forward 1x128 activation groups re-quantized as 128x1 for the backward
 *     pass: "英伟达破解AI训练效率难题" (163.com), section 五.
 *   - Mismatch metric token-mult-prob-error = (1/n) sum_i exp|logp_train_i -
 *     logp_infer_i|: nmedialink.com page, section "FP8面临的关键挑战：数值分歧".
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   E4M3 is the OCP "fn" format (bias 7, max 448, NaN 0x7F/0xFF, no inf);
 *   encode = round to nearest, ties to the even code, saturating at +-448,
 *   sign of zero kept; scale s = amax/448 as an IEEE binary32 division, and
 *   s = 1 when amax = 0; codes q = E4(fl32(x / s)); the 128x1 groups are
 *   re-quantized from the saved FP8 1x128 values v = fl32(D4(q) * s_row).
 *
 * Build with -O2 -fno-fast-math -ffp-contract=off so that every float
 * operation below is one IEEE binary32/binary64 operation with
 * round-to-nearest-even, in the order written.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* E4M3 codec                                                                */
/* ------------------------------------------------------------------------ */

/* Decode one E4M3 code from its bit fields: sign s (bit 7), exponent e
 * (bits 6..3, bias 7), mantissa m (bits 2..0).  e == 0 is subnormal,
 * m * 2^-9; e == 15 with m == 7 is NaN; everything else is normal,
 * (1 + m/8) * 2^(e-7). */
double jo_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

static double g_dec[256];
static int g_dec_ready = 0;
void jo_init(void);

static void dec_init(void)
{
    if (g_dec_ready)
        return;
    jo_init();
}

/* Fill the decode table; the loader calls this once before any threads. */
void jo_init(void)
{
    if (g_dec_ready)
        return;
    for (int c = 0; c < 256; ++c)
        g_dec[c] = jo_e4m3_decode((uint8_t)c);
    g_dec_ready = 1;
}

/* Encode a finite binary32 value: the non-negative code 0x00..0x7E whose
 * value is nearest to |v| (searched exhaustively, distances in binary64),
 * ties to the code with an even bit pattern, |v| >= 448 saturating to 0x7E;
 * then the sign bit of v is ORed in (so -0 and negative values that round to
 * zero give 0x80). */
uint8_t jo_e4m3_encode(float v)
{
    dec_init();
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0)
        return (uint8_t)(0x7E | sign);
    int best = 0;
    double bestd = fabs(g_dec[0] - a);
    for (int c = 1; c <= 0x7E; ++c) {
        double d = fabs(g_dec[c] - a);
        if (d < bestd) {
            bestd = d;
            best = c;
        } else if (d == bestd && (c & 1) == 0) {
            best = c; /* exact tie between neighbours: keep the even code */
        }
    }
    return (uint8_t)(best | sign);
}

/* Encode n values (same rule as jo_e4m3_encode). */
void jo_e4m3_encode_n(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = jo_e4m3_encode(v[i]);
}

/* ------------------------------------------------------------------------ */
/* Group scale and one-group quantization                                   */
/* ------------------------------------------------------------------------ */

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* s = amax / 448 (binary32 division), 1 when the group is all zero. */
float jo_group_scale(float amax)
{
    if (amax == 0.0f)
        return 1.0f;
    return amax / 448.0f;
}

/* Quantize n values vals[0], vals[stride], ... : returns the scale and
 * writes code i to codes[i * cstride]. */
static float quant_group(const float *vals, int64_t stride, int64_t n,
                         uint8_t *codes, int64_t cstride)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(vals[i * stride]);
        if (a > amax)
            amax = a;
    }
    float s = jo_group_scale(amax);
    for (int64_t i = 0; i < n; ++i) {
        float t = vals[i * stride] / s;
        codes[i * cstride] = jo_e4m3_encode(t);
    }
    return s;
}

/* ------------------------------------------------------------------------ */
/* The three groupings                                                      */
/* ------------------------------------------------------------------------ */

/* 1x128 groups along the last axis of x[M][K] (BF16 bits).
 * q[M][K] codes; s[kb * M + m] is the scale of row m, columns
 * 128*kb .. 128*kb+127.  Rows [m0, m1) only. */
void jo_quant_act_1x128(const uint16_t *x, int64_t M, int64_t K, uint8_t *q,
                        float *s, int64_t m0, int64_t m1)
{
    float g[128];
    int64_t Kb = K / 128;
    for (int64_t m = m0; m < m1; ++m)
        for (int64_t kb = 0; kb < Kb; ++kb) {
            for (int i = 0; i < 128; ++i)
                g[i] = bf16_to_f32(x[m * K + kb * 128 + i]);
            s[kb * M + m] = quant_group(g, 1, 128, q + m * K + kb * 128, 1);
        }
}

/* 128x128 blocks of w[N][K] (BF16 bits).  q[N][K]; s[nb * Kb + kb].
 * Block rows [nb0, nb1) only. */
void jo_quant_w_128x128(const uint16_t *w, int64_t N, int64_t K, uint8_t *q,
                        float *s, int64_t nb0, int64_t nb1)
{
    (void)N;
    int64_t Kb = K / 128;
    float *g = (float *)malloc(sizeof(float) * 128 * 128);
    uint8_t *c = (uint8_t *)malloc(128 * 128);
    for (int64_t nb = nb0; nb < nb1; ++nb)
        for (int64_t kb = 0; kb < Kb; ++kb) {
            for (int r = 0; r < 128; ++r)
                for (int i = 0; i < 128; ++i)
                    g[r * 128 + i] =
                        bf16_to_f32(w[(nb * 128 + r) * K + kb * 128 + i]);
            s[nb * Kb + kb] = quant_group(g, 1, 128 * 128, c, 1);
            for (int r = 0; r < 128; ++r)
                memcpy(q + (nb * 128 + r) * K + kb * 128, c + r * 128, 128);
        }
    free(g);
    free(c);
}

/* 128x1 re-quantization along the token axis, from the saved 1x128 form
 * (q[M][K], s[kb * M + m]).  v[m][k] = fl32(D4(q[m][k]) * s[k/128][m]);
 * each column k, token block mb (tokens 128*mb .. 128*mb+127) is one group.
 * Output transposed: qT[k * M + m], sT[mb * K + k].  Columns [k0, k1). */
void jo_requant_128x1(const uint8_t *q, const float *s, int64_t M, int64_t K,
                      uint8_t *qT, float *sT, int64_t k0, int64_t k1)
{
    dec_init();
    float g[128];
    int64_t Mb = M / 128;
    for (int64_t k = k0; k < k1; ++k)
        for (int64_t mb = 0; mb < Mb; ++mb) {
            for (int i = 0; i < 128; ++i) {
                int64_t m = mb * 128 + i;
                float d = (float)g_dec[q[m * K + k]];
                g[i] = d * s[(k / 128) * M + m];
            }
            sT[mb * K + k] =
                quant_group(g, 1, 128, qT + k * M + mb * 128, 1);
        }
}

/* ------------------------------------------------------------------------ */
/* SwiGLU with the 1x128 quantization of its output fused                   */
/* ------------------------------------------------------------------------ */
/* The pages fuse the quantization into the operator that produces a linear
 * layer's input, so that the saved activation is FP8 straight away ("英伟达
 * 破解AI训练效率难题" (163.com), section 三; "Jet-RL ..." (gist.science),
 * "Quantisierungsschema").  For the MLP's down projection that operator is
 * SwiGLU, h = silu(gate) * up.  The pages give no arithmetic for it; the
 * reading here is a fully specified binary32 evaluation (below), after which
 * the 128-wide groups of h are quantized exactly as activations are, from
 * the binary32 values (no BF16 rounding of h in between). */

/* e^x in binary32 for x in [-104, 80], by Cody-Waite argument reduction
 * x = n ln2 + r (ln 2 split into a 16-bit head and a rounded tail, both
 * products taken with fused multiply-adds), |r| <= ln2 / 2, the Taylor
 * polynomial of e^r to degree 7 in Horner form (coefficients RN(1/k!)),
 * and the scaling by 2^n as two exact powers of two, 2^(n/2) and
 * 2^(n - n/2) (C division, truncating), so that the only rounding of the
 * scaling is the final product's. */
static float pow2i(int k) /* 2^k for -126 <= k <= 127 */
{
    uint32_t u = (uint32_t)(k + 127) << 23;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

float jo_exp_f32(float x)
{
    const float log2e = 0x1.715476p+0f;
    const float ln2_hi = 0x1.62e4p-1f;
    const float ln2_lo = 0x1.7f7d1cp-20f;
    float n = rintf(x * log2e);
    float r = fmaf(n, -ln2_hi, x);
    r = fmaf(n, -ln2_lo, r);
    float p = 0x1.a01a02p-13f;          /* 1/7! */
    p = fmaf(p, r, 0x1.6c16c2p-10f);    /* 1/6! */
    p = fmaf(p, r, 0x1.111112p-7f);     /* 1/5! */
    p = fmaf(p, r, 0x1.555556p-5f);     /* 1/4! */
    p = fmaf(p, r, 0x1.555556p-3f);     /* 1/3! */
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    int ni = (int)n;
    int n1 = ni / 2;
    p = p * pow2i(n1);
    p = p * pow2i(ni - n1);
    return p;
}

/* silu(g) = g / (1 + e^-g) in binary32.  For g < -80 the true value is
 * below 1.5e-33 in magnitude and is taken as g * 0 (a signed zero).
 * Otherwise the exponent -g is clamped below at -104 (where e^-g no longer
 * changes 1 + e^-g), d = 1 + e^-g, and 1/d is taken from the bit-pattern
 * seed 0x7EF311C7 - bits(d) refined by three Newton-Raphson steps
 * y <- y + y (1 - d y) (fused multiply-adds); silu = g * (1/d). */
float jo_silu_f32(float g)
{
    if (g < -80.0f)
        return g * 0.0f;
    float x = -g;
    if (x < -104.0f)
        x = -104.0f;
    float d = 1.0f + jo_exp_f32(x);
    uint32_t b;
    memcpy(&b, &d, sizeof b);
    b = 0x7EF311C7u - b;
    float y;
    memcpy(&y, &b, sizeof y);
    for (int i = 0; i < 3; ++i)
        y = fmaf(fmaf(-d, y, 1.0f), y, y);
    return g * y;
}

/* h[m][f] = fl32(silu(gate[m][f]) * up[m][f]) for gate, up BF16 with rows
 * ld elements apart (gate[m][f] = g[m * ld + f], up likewise from u), then
 * 1x128 groups of h along f: q[M][F] codes, s[fb * M + m] scales.  Rows
 * [m0, m1) only. */
void jo_swiglu_quant_1x128(const uint16_t *g, const uint16_t *u, int64_t ld,
                           int64_t M, int64_t F, uint8_t *q, float *s,
                           int64_t m0, int64_t m1)
{
    float h[128];
    int64_t Fb = F / 128;
    for (int64_t m = m0; m < m1; ++m)
        for (int64_t fb = 0; fb < Fb; ++fb) {
            for (int i = 0; i < 128; ++i) {
                int64_t at = m * ld + fb * 128 + i;
                h[i] = jo_silu_f32(bf16_to_f32(g[at])) * bf16_to_f32(u[at]);
            }
            s[fb * M + m] = quant_group(h, 1, 128, q + m * F + fb * 128, 1);
        }
}

/* ------------------------------------------------------------------------ */
/* RMSNorm with the 1x128 quantization of its output fused                  */
/* ------------------------------------------------------------------------ */
/* The pages' system runs fused activation and RMSNorm operators
 * ("Jet-RL ..." (gist.science), "Implementierung") and quantizes a linear
 * layer's input in the operator that produces it ("英伟达破解AI训练效率难题"
 * (163.com), section 五).  RMSNorm produces the inputs of the q/k/v and the
 * gate/up projections.  The pages give no arithmetic for it; the reading here
 * is RMSNorm y = x * g / sqrt(mean(x^2) + eps) evaluated in binary32 by one
 * fixed sequence of IEEE operations, after which the 128-wide groups of the
 * binary32 y are quantized exactly as activations are (no BF16 rounding of y
 * in between):
 *   - sum of squares of a row of K values: 32 partial sums; partial l adds,
 *     in this order, the squares of the elements 8 (32 j + l) + t for
 *     j = 0, 1, ... (while 8 (32 j + l) < K) and t = 0 .. 7, one binary32
 *     rounding per addition (the square of a BF16 value is exact in
 *     binary32); then five butterfly levels d = 16, 8, 4, 2, 1 replace
 *     partial l by partial l + partial (l xor d) (every partial ends equal,
 *     addition being commutative) and ss is partial 0;
 *   - ms = fl32(ss / K), v = fl32(ms + eps), r = fl32(1 / fl32(sqrt(v)))
 *     (IEEE division and square root), r = 0 when v == 0;
 *   - y_k = fl32(fl32(x_k * r) * g_k).
 * Rows whose sum of squares overflows binary32 are outside the contract. */
static float rms_factor(const uint16_t *xr, int64_t K, float eps)
{
    float part[32];
    for (int l = 0; l < 32; ++l) {
        float acc = 0.0f;
        for (int64_t j = 0; 8 * (32 * j + l) < K; ++j)
            for (int t = 0; t < 8; ++t) {
                float v = bf16_to_f32(xr[8 * (32 * j + l) + t]);
                acc = acc + v * v;
            }
        part[l] = acc;
    }
    for (int d = 16; d >= 1; d /= 2) {
        float nxt[32];
        for (int l = 0; l < 32; ++l)
            nxt[l] = part[l] + part[l ^ d];
        memcpy(part, nxt, sizeof part);
    }
    float ms = part[0] / (float)K;
    float v = ms + eps;
    if (v == 0.0f)
        return 0.0f;
    float root = sqrtf(v);
    return 1.0f / root;
}

/* y[m][k] (binary32) of rows [m0, m1) of x[M][K] with gain g[K] (BF16). */
void jo_rmsnorm_f32(const uint16_t *x, const uint16_t *g, int64_t M, int64_t K,
                    float eps, float *y, int64_t m0, int64_t m1)
{
    (void)M;
    for (int64_t m = m0; m < m1; ++m) {
        float r = rms_factor(x + m * K, K, eps);
        for (int64_t k = 0; k < K; ++k) {
            float t = bf16_to_f32(x[m * K + k]) * r;
            y[m * K + k] = t * bf16_to_f32(g[k]);
        }
    }
}

/* RMSNorm of x[M][K] with gain g[K] (BF16 bits), then 1x128 groups of y:
 * q[M][K] codes, s[kb * M + m] scales.  Rows [m0, m1) only. */
void jo_rmsnorm_quant_1x128(const uint16_t *x, const uint16_t *g, int64_t M,
                            int64_t K, float eps, uint8_t *q, float *s,
                            int64_t m0, int64_t m1)
{
    float y[128];
    int64_t Kb = K / 128;
    for (int64_t m = m0; m < m1; ++m) {
        float r = rms_factor(x + m * K, K, eps);
        for (int64_t kb = 0; kb < Kb; ++kb) {
            for (int i = 0; i < 128; ++i) {
                int64_t k = kb * 128 + i;
                float t = bf16_to_f32(x[m * K + k]) * r;
                y[i] = t * bf16_to_f32(g[k]);
            }
            s[kb * M + m] = quant_group(y, 1, 128, q + m * K + kb * 128, 1);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* GEMMs: binary64 product of the dequantized operands                       */
/* ------------------------------------------------------------------------ */

/* Row-sampled GEMM  out[r][j] = sum_c A(rows[r], c) * B(j, c), r in [r0, r1),
 * every dequantized operand and every product and sum in binary64.
 *   fwd   (kind 0): A = X  [M][K],  scale sx [c/128][i];
 *                   B(j=n, c=k) = W[n][k],  scale sw [n/128][k/128].
 *   dgrad (kind 1): A = dY [M][N],  scale sdy[c/128][i];
 *                   B(j=k, c=n) = W[n][k],  scale sw [n/128][k/128].
 *   wgrad (kind 2): A = dYT[N][M],  scale sdyT[c/128][i];
 *                   B(j=k, c=m) = XT[k][m], scale sxT[m/128][k].
 * nrows_a is the row count of A (the stride of its scale array),
 * ncols_out the output width, depth the contraction length. */
static double deq_a(const uint8_t *qa, const float *sa, int64_t nrows_a,
                    int64_t depth, int64_t i, int64_t c)
{
    return g_dec[qa[i * depth + c]] * (double)sa[(c / 128) * nrows_a + i];
}

static double deq_b(int kind, const uint8_t *qb, const float *sb,
                    int64_t ncols_out, int64_t depth, int64_t j, int64_t c)
{
    switch (kind) {
    case 0:
        return g_dec[qb[j * depth + c]] *
               (double)sb[(j / 128) * (depth / 128) + c / 128];
    case 1:
        return g_dec[qb[c * ncols_out + j]] *
               (double)sb[(c / 128) * (ncols_out / 128) + j / 128];
    default:
        return g_dec[qb[j * depth + c]] * (double)sb[(c / 128) * ncols_out + j];
    }
}

static void gemm_rows(int kind, const uint8_t *qa, const float *sa,
                      const uint8_t *qb, const float *sb, int64_t nrows_a,
                      int64_t ncols_out, int64_t depth, const int64_t *rows,
                      int64_t r0, int64_t r1, double *out)
{
    dec_init();
    for (int64_t r = r0; r < r1; ++r) {
        int64_t i = rows[r];
        for (int64_t j = 0; j < ncols_out; ++j) {
            double acc = 0.0;
            for (int64_t c = 0; c < depth; ++c)
                acc += deq_a(qa, sa, nrows_a, depth, i, c) *
                       deq_b(kind, qb, sb, ncols_out, depth, j, c);
            out[r * ncols_out + j] = acc;
        }
    }
}

/* Y[r][n] = sum_k dq(X)[rows[r]][k] * dq(W)[n][k];  X [M][K], W [N][K]. */
void jo_gemm_fwd(const uint8_t *qx, const float *sx, const uint8_t *qw,
                 const float *sw, int64_t M, int64_t N, int64_t K,
                 const int64_t *rows, int64_t r0, int64_t r1, double *y)
{
    gemm_rows(0, qx, sx, qw, sw, M, N, K, rows, r0, r1, y);
}

/* dX[r][k] = sum_n dq(dY)[rows[r]][n] * dq(W)[n][k];  dY [M][N]. */
void jo_gemm_dgrad(const uint8_t *qdy, const float *sdy, const uint8_t *qw,
                   const float *sw, int64_t M, int64_t N, int64_t K,
                   const int64_t *rows, int64_t r0, int64_t r1, double *dx)
{
    gemm_rows(1, qdy, sdy, qw, sw, M, K, N, rows, r0, r1, dx);
}

/* dW[r][k] = sum_m dq(dYT)[rows[r]][m] * dq(XT)[k][m];
 * dYT [N][M] with scales [M/128][N], XT [K][M] with scales [M/128][K]. */
void jo_gemm_wgrad(const uint8_t *qdyT, const float *sdyT, const uint8_t *qxT,
                   const float *sxT, int64_t M, int64_t N, int64_t K,
                   const int64_t *rows, int64_t r0, int64_t r1, double *dw)
{
    gemm_rows(2, qdyT, sdyT, qxT, sxT, N, K, M, rows, r0, r1, dw);
}

/* ------------------------------------------------------------------------ */
/* Mismatch metric                                                          */
/* ------------------------------------------------------------------------ */

/* (1/n) * sum_i exp(|a_i - b_i|), inputs widened to binary64. */
double jo_token_mult_prob_error(const float *a, const float *b, int64_t n)
{
    double sum = 0.0;
    for (int64_t i = 0; i < n; ++i)
        sum += exp(fabs((double)a[i] - (double)b[i]));
    return sum / (double)n;
}

/* Masked mismatch metric with per-token importance weights.
 * The importance weight of a token is the ratio of the training model's
 * probability of it to the rollout model's ("FP8-RL" article: the ratio of
 * the original to the compressed model's token probability), here
 * w_i = exp(a_i - b_i) with a = logp_train and b = logp_rollout, optionally
 * capped at `cap` (cap <= 0: no cap; the pages give no constant), and 0 for a
 * token outside the mask.  The metric is the token-mult-prob-error of the
 * nmedialink page over the masked tokens only:
 *   (sum over masked i of exp|a_i - b_i|) / count.
 * mask == NULL counts every token.  *count receives the number of masked
 * tokens; with none the metric is NaN.  All arithmetic in binary64. */
double jo_token_mismatch_masked(const float *a, const float *b, const uint8_t *mask,
                                int64_t n, double cap, double *w, int64_t *count)
{
    double sum = 0.0;
    int64_t c = 0;
    for (int64_t i = 0; i < n; ++i) {
        const int on = mask == NULL || mask[i] != 0;
        const double d = (double)a[i] - (double)b[i];
        if (on) {
            double wi = exp(d);
            if (cap > 0.0 && wi > cap) wi = cap;
            w[i] = wi;
            sum += exp(fabs(d));
            ++c;
        } else {
            w[i] = 0.0;
        }
    }
    *count = c;
    return c > 0 ? sum / (double)c : NAN;
}

/* ------------------------------------------------------------------------ */
/* FP8 KV cache with the scales recalibrated after each model update         */
/* ------------------------------------------------------------------------ */
/* The FP8-RL article extends the compressed format to the KV cache: the
 * scale factors are calibrated again after every model update and the cache
 * entries are stored compressed with them ("FP8-RL" article (m.66260.cn), the
 * KV-cache paragraph; the nmedialink page, "FP8探索新维度：KV缓存与注意力机制赋能").
 * They give no granularity.  Reading: one binary32 scale per KV head (for K
 * and for V separately), s_h = amax_h / 448 over the calibration tokens
 * (all tokens and all D channels of head h; s_h = 1 when amax_h = 0), the
 * group rule's scale; entries written afterwards are E4(fl32(x / s_h)),
 * saturating at +-448 when they exceed the calibrated range. */

/* scale[h] for x[T][H][D] (BF16 bits). */
void jo_kv_calibrate(const uint16_t *x, int64_t T, int64_t H, int64_t D, float *scale)
{
    for (int64_t h = 0; h < H; ++h) {
        float amax = 0.0f;
        for (int64_t t = 0; t < T; ++t)
            for (int64_t d = 0; d < D; ++d) {
                float a = fabsf(bf16_to_f32(x[(t * H + h) * D + d]));
                if (a > amax)
                    amax = a;
            }
        scale[h] = jo_group_scale(amax);
    }
}

/* cache[slot[t]][h][d] = E4(fl32(x[t][h][d] / scale[h])) for the T new
 * entries x[T][H][D] (BF16 bits); cache has S slots of H x D codes.  A slot
 * outside [0, S) is skipped. */
void jo_kv_cache_write(const uint16_t *x, const float *scale, const int64_t *slot, int64_t T,
                       int64_t H, int64_t D, uint8_t *cache, int64_t S)
{
    for (int64_t t = 0; t < T; ++t) {
        if (slot[t] < 0 || slot[t] >= S)
            continue;
        for (int64_t h = 0; h < H; ++h)
            for (int64_t d = 0; d < D; ++d) {
                float v = bf16_to_f32(x[(t * H + h) * D + d]);
                cache[(slot[t] * H + h) * D + d] = jo_e4m3_encode(v / scale[h]);
            }
    }
}
