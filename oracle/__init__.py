"""CPU oracle for the unified-precision FP8 linear layer (Jet-RL).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product library (``fp8_block_quantized_gb300``) never imports it and has no
fallback to it.

The arithmetic lives in ``jet_oracle.c`` (plain C, built with
``-O2 -fno-fast-math -ffp-contract=off``); this module only builds it, loads it
with ctypes and marshals numpy arrays.  Row/column ranges are spread over
threads (ctypes releases the GIL during a foreign call); that split is over
independent output rows and changes no arithmetic.

Sources followed (page title and section):
  * quantization table (weights E4M3 [128,128], input activations and output
    gradients E4M3 [1,128], FP32 block scales): "NVIDIA强化学习加速实操：10分钟
    提升2倍训练效率", section "为什么FP8适配线性层？";
  * 1x128 activations, 128x128 weights, FP8 DGrad/WGrad with 1x128 and 128x1
    groups: "Jet-RL: Enabling On-Policy FP8 Reinforcement Learning with Unified
    Training and Rollout Precision Flow" (gist.science), "Quantisierungsschema";
  * 1x128 forward groups re-quantized as 128x1 in backward: "英伟达破解AI训练
    效率难题" (163.com), section 五;
  * token-mult-prob-error: nmedialink page, section "FP8面临的关键挑战：数值分歧";
  * importance weights (ratio of the original to the compressed model's token
    probability): FP8-RL article (m.66260.cn), paragraph on error correction;
    importance sampling combined with FP8: nmedialink page, section
    "重要抽样技术：提升RL精度的尖兵".

Every function here is pinned by ``tests/test_oracle_*.py`` against facts the
pages or mathematics fix (no function is "parity unpinned").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "jet_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
          "-std=c11", "-Wall"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``jet_oracle.c`` into ``_build/liboracle.so`` (gcc, portable C)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int64
        lib.jo_init.restype = None
        lib.jo_e4m3_decode.restype = ctypes.c_double
        lib.jo_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.jo_e4m3_encode.restype = ctypes.c_uint8
        lib.jo_e4m3_encode.argtypes = [ctypes.c_float]
        lib.jo_e4m3_encode_n.argtypes = [P, I, P]
        lib.jo_e4m3_encode_n.restype = None
        lib.jo_group_scale.restype = ctypes.c_float
        lib.jo_group_scale.argtypes = [ctypes.c_float]
        lib.jo_quant_act_1x128.argtypes = [P, I, I, P, P, I, I]
        lib.jo_quant_w_128x128.argtypes = [P, I, I, P, P, I, I]
        lib.jo_requant_128x1.argtypes = [P, P, I, I, P, P, I, I]
        lib.jo_exp_f32.argtypes = [ctypes.c_float]
        lib.jo_exp_f32.restype = ctypes.c_float
        lib.jo_silu_f32.argtypes = [ctypes.c_float]
        lib.jo_silu_f32.restype = ctypes.c_float
        lib.jo_swiglu_quant_1x128.argtypes = [P, P, I, I, I, P, P, I, I]
        lib.jo_rmsnorm_f32.argtypes = [P, P, I, I, ctypes.c_float, P, I, I]
        lib.jo_rmsnorm_f32.restype = None
        lib.jo_rmsnorm_quant_1x128.argtypes = [P, P, I, I, ctypes.c_float, P, P, I, I]
        lib.jo_rmsnorm_quant_1x128.restype = None
        lib.jo_kv_calibrate.argtypes = [P, I, I, I, P]
        lib.jo_kv_cache_write.argtypes = [P, P, P, I, I, I, P, I]
        for f in (lib.jo_gemm_fwd, lib.jo_gemm_dgrad, lib.jo_gemm_wgrad):
            f.argtypes = [P, P, P, P, I, I, I, P, I, I, P]
            f.restype = None
        lib.jo_token_mult_prob_error.restype = ctypes.c_double
        lib.jo_token_mult_prob_error.argtypes = [P, P, I]
        lib.jo_token_mismatch_masked.restype = ctypes.c_double
        lib.jo_token_mismatch_masked.argtypes = [P, P, P, I, ctypes.c_double, P,
                                                 ctypes.POINTER(ctypes.c_int64)]
        lib.jo_init()
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _threads(nthreads):
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    return max(1, int(nthreads))


def _split(n: int, parts: int):
    parts = max(1, min(parts, n)) if n > 0 else 1
    per = (n + parts - 1) // parts
    return [(i * per, min(n, (i + 1) * per)) for i in range(parts)
            if i * per < min(n, (i + 1) * per)]


def _run(fn, n, nthreads):
    ranges = _split(n, _threads(nthreads))
    if len(ranges) <= 1:
        for a, b in ranges:
            fn(a, b)
        return
    with ThreadPoolExecutor(len(ranges)) as ex:
        list(ex.map(lambda r: fn(*r), ranges))


# --------------------------------------------------------------------------
# E4M3 codec
# --------------------------------------------------------------------------

def e4m3_decode(code: int) -> float:
    """Value of one E4M3 code (NaN for 0x7F / 0xFF)."""
    return _load().jo_e4m3_decode(int(code) & 0xFF)


def e4m3_decode_table() -> np.ndarray:
    """float64[256]: the value of every code."""
    lib = _load()
    return np.array([lib.jo_e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(v) -> np.ndarray:
    """Encode finite float32 values (any shape) to uint8 codes."""
    lib = _load()
    a = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint8)
    lib.jo_e4m3_encode_n(_ptr(a), a.size, _ptr(out))
    return out


def group_scale(amax: float) -> np.float32:
    """s = amax / 448 in binary32 (1 when amax == 0)."""
    return np.float32(_load().jo_group_scale(float(np.float32(amax))))


# --------------------------------------------------------------------------
# Quantizers
# --------------------------------------------------------------------------

def _as_bf16_bits(x) -> np.ndarray:
    a = np.asarray(x)
    if a.dtype != np.uint16:
        raise TypeError("BF16 tensors are passed as their uint16 bit patterns")
    return np.ascontiguousarray(a)


def quant_act_1x128(x_bits, nthreads=None):
    """1x128 groups of x[M][K] (BF16 bits) -> (q uint8 [M,K], s float32 [K/128, M])."""
    lib = _load()
    x = _as_bf16_bits(x_bits)
    M, K = x.shape
    if K % 128:
        raise ValueError("K must be a multiple of 128")
    q = np.empty((M, K), np.uint8)
    s = np.empty((K // 128, M), np.float32)
    _run(lambda a, b: lib.jo_quant_act_1x128(_ptr(x), M, K, _ptr(q), _ptr(s), a, b),
         M, nthreads)
    return q, s


def exp_f32(x):
    """The binary32 e^x of the fused SwiGLU quantizer (x in [-104, 80]), elementwise.
    Pinned against binary64 exp (within 1 ulp where the result is normal)."""
    lib = _load()
    return np.array([lib.jo_exp_f32(float(v)) for v in np.asarray(x, np.float32).ravel()],
                    np.float32).reshape(np.shape(x))


def silu_f32(g):
    """The binary32 silu(g) = g / (1 + e^-g) of the fused SwiGLU quantizer, elementwise."""
    lib = _load()
    return np.array([lib.jo_silu_f32(float(v)) for v in np.asarray(g, np.float32).ravel()],
                    np.float32).reshape(np.shape(g))


def swiglu_quant_1x128(gate_bits, up_bits, nthreads=None):
    """h = silu(gate) * up in binary32, then 1x128 groups of h ->
    (q uint8 [M,F], s float32 [F/128, M]).  gate, up: BF16 bits [M,F]."""
    lib = _load()
    g = _as_bf16_bits(gate_bits)
    u = _as_bf16_bits(up_bits)
    if g.shape != u.shape:
        raise ValueError("gate and up must have the same shape")
    M, F = g.shape
    if F % 128:
        raise ValueError("F must be a multiple of 128")
    q = np.empty((M, F), np.uint8)
    s = np.empty((F // 128, M), np.float32)
    _run(lambda a, b: lib.jo_swiglu_quant_1x128(_ptr(g), _ptr(u), F, M, F, _ptr(q), _ptr(s),
                                                a, b), M, nthreads)
    return q, s


def _rms_args(x_bits, g_bits, eps):
    x = _as_bf16_bits(x_bits)
    g = _as_bf16_bits(g_bits).reshape(-1)
    if x.ndim != 2 or g.size != x.shape[1]:
        raise ValueError("x must be [M, K] and g [K]")
    if not (np.isfinite(eps) and eps >= 0):
        raise ValueError("eps must be finite and >= 0")
    return x, np.ascontiguousarray(g), np.float32(eps)


def rmsnorm_f32(x_bits, g_bits, eps, nthreads=None):
    """The binary32 RMSNorm y = x * g / sqrt(mean(x^2) + eps) of the fused
    RMSNorm quantizer (its fixed order of operations; see jet_oracle.c):
    y float32 [M, K].  x: BF16 bits [M, K]; g: BF16 bits [K]."""
    lib = _load()
    x, g, e = _rms_args(x_bits, g_bits, eps)
    M, K = x.shape
    y = np.empty((M, K), np.float32)
    _run(lambda a, b: lib.jo_rmsnorm_f32(_ptr(x), _ptr(g), M, K, float(e), _ptr(y), a, b),
         M, nthreads)
    return y


def rmsnorm_quant_1x128(x_bits, g_bits, eps, nthreads=None):
    """RMSNorm of x (binary32, as rmsnorm_f32), then 1x128 groups of y ->
    (q uint8 [M,K], s float32 [K/128, M])."""
    lib = _load()
    x, g, e = _rms_args(x_bits, g_bits, eps)
    M, K = x.shape
    if K % 128:
        raise ValueError("K must be a multiple of 128")
    q = np.empty((M, K), np.uint8)
    s = np.empty((K // 128, M), np.float32)
    _run(lambda a, b: lib.jo_rmsnorm_quant_1x128(_ptr(x), _ptr(g), M, K, float(e), _ptr(q),
                                                 _ptr(s), a, b), M, nthreads)
    return q, s


def quant_w_128x128(w_bits, nthreads=None):
    """128x128 blocks of w[N][K] (BF16 bits) -> (q uint8 [N,K], s float32 [N/128, K/128])."""
    lib = _load()
    w = _as_bf16_bits(w_bits)
    N, K = w.shape
    if N % 128 or K % 128:
        raise ValueError("N and K must be multiples of 128")
    q = np.empty((N, K), np.uint8)
    s = np.empty((N // 128, K // 128), np.float32)
    _run(lambda a, b: lib.jo_quant_w_128x128(_ptr(w), N, K, _ptr(q), _ptr(s), a, b),
         N // 128, nthreads)
    return q, s


def requant_128x1(q, s, nthreads=None):
    """128x1 re-quantization of the saved 1x128 form.

    q uint8 [M,K], s float32 [K/128, M] -> (qT uint8 [K,M], sT float32 [M/128, K]).
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.float32)
    M, K = q.shape
    if M % 128 or K % 128 or s.shape != (K // 128, M):
        raise ValueError("need M, K multiples of 128 and s of shape [K/128, M]")
    qT = np.empty((K, M), np.uint8)
    sT = np.empty((M // 128, K), np.float32)
    _run(lambda a, b: lib.jo_requant_128x1(_ptr(q), _ptr(s), M, K, _ptr(qT), _ptr(sT), a, b),
         K, nthreads)
    return qT, sT


# --------------------------------------------------------------------------
# GEMMs (binary64 product of the dequantized operands)
# --------------------------------------------------------------------------

def _gemm(fn, qa, sa, qb, sb, M, N, K, nout_rows_total, ncols, rows, nthreads):
    qa = np.ascontiguousarray(qa, np.uint8)
    qb = np.ascontiguousarray(qb, np.uint8)
    sa = np.ascontiguousarray(sa, np.float32)
    sb = np.ascontiguousarray(sb, np.float32)
    if rows is None:
        rows = np.arange(nout_rows_total, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= nout_rows_total):
        raise IndexError("row index out of range")
    out = np.empty((rows.size, ncols), np.float64)
    _run(lambda a, b: fn(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), M, N, K,
                         _ptr(rows), a, b, _ptr(out)), rows.size, nthreads)
    return out


def gemm_fwd(qx, sx, qw, sw, rows=None, nthreads=None):
    """Y = dq(X) . dq(W)^T in binary64; X [M,K] (sx [K/128,M]), W [N,K] (sw [N/128,K/128]).

    ``rows`` selects output rows (default all); returns float64 [len(rows), N].
    """
    M, K = np.shape(qx)
    N = np.shape(qw)[0]
    assert np.shape(qw)[1] == K and np.shape(sx) == (K // 128, M)
    assert np.shape(sw) == (N // 128, K // 128)
    return _gemm(_load().jo_gemm_fwd, qx, sx, qw, sw, M, N, K, M, N, rows, nthreads)


def gemm_fwd_grouped(qx, sx, qw, sw, offsets, nthreads=None):
    """Grouped forward product of expert linears: for every expert e,
    Y[o_e:o_{e+1}] = dq(X[o_e:o_{e+1}]) . dq(W_e)^T in binary64.

    X [Mtot,K] holds the tokens of all experts in expert order (sx [K/128,
    Mtot]); W [E,N,K] the experts' weights (sw [E,N/128,K/128]); offsets
    [E+1] the experts' first rows (offsets[0] = 0, non-decreasing,
    offsets[E] = Mtot).  Each expert's rows are the plain forward product of
    its own tokens and weights (its definition and pins are gemm_fwd's)."""
    qw = np.asarray(qw)
    sw = np.asarray(sw)
    E, N, K = qw.shape
    off = np.asarray(offsets, np.int64)
    assert off.shape == (E + 1,) and off[0] == 0 and (np.diff(off) >= 0).all()
    assert np.shape(qx) == (off[-1], K) and np.shape(sx) == (K // 128, off[-1])
    assert sw.shape == (E, N // 128, K // 128)
    out = np.zeros((int(off[-1]), N), np.float64)
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            out[a:b] = gemm_fwd(np.ascontiguousarray(qx[a:b]), np.ascontiguousarray(sx[:, a:b]),
                                qw[e], sw[e], nthreads=nthreads)
    return out


def gemm_dgrad_grouped(qdy, sdy, qw, sw, offsets, nthreads=None):
    """Grouped DGrad of expert linears: for every expert e,
    dX[o_e:o_{e+1}] = dq(dY[o_e:o_{e+1}]) . dq(W_e) in binary64.

    dY [Mtot,N] holds the output gradients of all experts' tokens in expert
    order (sdy [N/128, Mtot]); W [E,N,K] (sw [E,N/128,K/128]); offsets as in
    gemm_fwd_grouped.  Each expert's rows are the plain DGrad product of its
    own rows and weights."""
    qw = np.asarray(qw)
    sw = np.asarray(sw)
    E, N, K = qw.shape
    off = np.asarray(offsets, np.int64)
    assert off.shape == (E + 1,) and off[0] == 0 and (np.diff(off) >= 0).all()
    assert np.shape(qdy) == (off[-1], N) and np.shape(sdy) == (N // 128, off[-1])
    assert sw.shape == (E, N // 128, K // 128)
    out = np.zeros((int(off[-1]), K), np.float64)
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            out[a:b] = gemm_dgrad(np.ascontiguousarray(qdy[a:b]),
                                  np.ascontiguousarray(sdy[:, a:b]), qw[e], sw[e],
                                  nthreads=nthreads)
    return out


def gemm_wgrad_grouped(qdyT, sdyT, qxT, sxT, offsets, nthreads=None):
    """Grouped WGrad of expert linears: for every expert e, the contraction
    over its own tokens, dW_e = dq(dYT[:, o_e:o_{e+1}]) . dq(XT[:, o_e:o_{e+1}])^T
    in binary64, from the 128x1 (transposed) forms of the expert-ordered
    tensors: dYT [N,Mtot] (sdyT [Mtot/128, N]), XT [K,Mtot] (sxT [Mtot/128, K]).
    The 128-token groups of those forms may not straddle two experts, so every
    offset is a multiple of 128 (experts padded to whole token blocks).
    Returns float64 [E, N, K]; an expert without tokens gets zeros."""
    off = np.asarray(offsets, np.int64)
    E = off.size - 1
    N, Mt = np.shape(qdyT)
    K = np.shape(qxT)[0]
    if off[0] != 0 or off[-1] != Mt or (np.diff(off) < 0).any() or (off % 128).any():
        raise ValueError("offsets must run from 0 to Mtot, non-decreasing, in multiples of 128")
    assert np.shape(qxT) == (K, Mt) and np.shape(sdyT) == (Mt // 128, N)
    assert np.shape(sxT) == (Mt // 128, K)
    out = np.zeros((E, N, K), np.float64)
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            out[e] = gemm_wgrad(np.ascontiguousarray(qdyT[:, a:b]),
                                np.ascontiguousarray(sdyT[a // 128:b // 128]),
                                np.ascontiguousarray(qxT[:, a:b]),
                                np.ascontiguousarray(sxT[a // 128:b // 128]), nthreads=nthreads)
    return out


def gemm_dgrad(qdy, sdy, qw, sw, rows=None, nthreads=None):
    """dX = dq(dY) . dq(W) in binary64; dY [M,N] (sdy [N/128,M]), W [N,K]."""
    M, N = np.shape(qdy)
    K = np.shape(qw)[1]
    assert np.shape(qw)[0] == N and np.shape(sdy) == (N // 128, M)
    assert np.shape(sw) == (N // 128, K // 128)
    return _gemm(_load().jo_gemm_dgrad, qdy, sdy, qw, sw, M, N, K, M, K, rows, nthreads)


def gemm_wgrad(qdyT, sdyT, qxT, sxT, rows=None, nthreads=None):
    """dW = dq(dYT) . dq(XT)^T in binary64; dYT [N,M] (sdyT [M/128,N]), XT [K,M] (sxT [M/128,K])."""
    N, M = np.shape(qdyT)
    K = np.shape(qxT)[0]
    assert np.shape(qxT)[1] == M and np.shape(sdyT) == (M // 128, N)
    assert np.shape(sxT) == (M // 128, K)
    return _gemm(_load().jo_gemm_wgrad, qdyT, sdyT, qxT, sxT, M, N, K, N, K, rows, nthreads)


# --------------------------------------------------------------------------
# Metric
# --------------------------------------------------------------------------

def token_mult_prob_error(logp_train, logp_infer) -> float:
    """(1/n) * sum_i exp(|logp_train_i - logp_infer_i|), binary64."""
    a = np.ascontiguousarray(logp_train, np.float32).reshape(-1)
    b = np.ascontiguousarray(logp_infer, np.float32).reshape(-1)
    if a.size != b.size or a.size == 0:
        raise ValueError("need two non-empty vectors of equal length")
    return float(_load().jo_token_mult_prob_error(_ptr(a), _ptr(b), a.size))


def token_mismatch_masked(logp_train, logp_rollout, mask=None, cap: float = 0.0):
    """(metric, count, w): the token-mult-prob-error over the masked tokens,
    their number, and the per-token importance weights
    w_i = min(exp(logp_train_i - logp_rollout_i), cap) (cap <= 0: no cap),
    0 outside the mask; binary64.  mask=None counts every token."""
    a = np.ascontiguousarray(logp_train, np.float32).reshape(-1)
    b = np.ascontiguousarray(logp_rollout, np.float32).reshape(-1)
    if a.size != b.size:
        raise ValueError("need two vectors of equal length")
    m = None if mask is None else np.ascontiguousarray(mask, np.uint8).reshape(-1)
    if m is not None and m.size != a.size:
        raise ValueError("mask length differs")
    w = np.empty(a.size, np.float64)
    count = ctypes.c_int64(0)
    metric = _load().jo_token_mismatch_masked(_ptr(a), _ptr(b), None if m is None else _ptr(m),
                                              a.size, float(cap), _ptr(w), ctypes.byref(count))
    return float(metric), int(count.value), w


def token_mismatch_per_sequence(logp_train, logp_rollout, seq_offsets, mask=None,
                                cap: float = 0.0):
    """(metrics [S], counts [S], w [n]): the masked token-mult-prob-error of
    every sequence s (tokens seq_offsets[s] .. seq_offsets[s+1]), its number
    of masked tokens, and the per-token importance weights, binary64.  Each
    sequence's figures are token_mismatch_masked over that sequence alone."""
    a = np.ascontiguousarray(logp_train, np.float32).reshape(-1)
    b = np.ascontiguousarray(logp_rollout, np.float32).reshape(-1)
    off = np.asarray(seq_offsets, np.int64)
    if off[0] != 0 or off[-1] != a.size or (np.diff(off) < 0).any():
        raise ValueError("offsets must run from 0 to n, non-decreasing")
    S = off.size - 1
    m = None if mask is None else np.ascontiguousarray(mask, np.uint8).reshape(-1)
    metrics = np.empty(S, np.float64)
    counts = np.empty(S, np.int64)
    w = np.empty(a.size, np.float64)
    for s in range(S):
        lo, hi = int(off[s]), int(off[s + 1])
        r, c, ws = token_mismatch_masked(a[lo:hi], b[lo:hi], None if m is None else m[lo:hi], cap)
        metrics[s], counts[s], w[lo:hi] = r, c, ws
    return metrics, counts, w


# --------------------------------------------------------------------------
# FP8 KV cache, scales recalibrated after each model update
# --------------------------------------------------------------------------

def kv_calibrate(x_bits):
    """Per-head scales s_h = amax_h / 448 (1 if amax_h = 0) of x [T, H, D]
    (BF16 bits): the calibration after a model update."""
    x = _as_bf16_bits(x_bits)
    T, H, D = x.shape
    s = np.empty(H, np.float32)
    _load().jo_kv_calibrate(_ptr(x), T, H, D, _ptr(s))
    return s


def kv_cache_write(x_bits, scale, slots, cache):
    """Write the new entries x [T, H, D] (BF16 bits) into ``cache`` [S, H, D]
    (uint8, modified in place) at rows ``slots`` [T] as E4(fl32(x / s_h));
    slots outside [0, S) are skipped.  Returns ``cache``."""
    x = _as_bf16_bits(x_bits)
    T, H, D = x.shape
    scale = np.ascontiguousarray(scale, np.float32)
    slots = np.ascontiguousarray(slots, np.int64)
    if not (cache.flags["C_CONTIGUOUS"] and cache.dtype == np.uint8):
        raise TypeError("cache must be a C-contiguous uint8 array")
    S = cache.shape[0]
    assert cache.shape == (S, H, D) and scale.shape == (H,) and slots.shape == (T,)
    _load().jo_kv_cache_write(_ptr(x), _ptr(scale), _ptr(slots), T, H, D, _ptr(cache), S)
    return cache
