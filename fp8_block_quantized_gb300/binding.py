"""Thin ctypes binding of the jet_fp8 C ABI (``include/jet_fp8.h``).

Argument marshalling only: every function here takes CUDA tensors, checks
their dtype/shape/device, and forwards the raw device pointers, sizes and the
current CUDA stream to the C entry point of the same name.  All quantization,
GEMM and reduction work happens in the library's kernels.  There is no CPU
fallback: if the library is missing or fails to load, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

STATUS = {0: "JET_OK", 1: "JET_ERR_NULL", 2: "JET_ERR_SHAPE", 3: "JET_ERR_ALIGN",
          4: "JET_ERR_CUDA", 5: "JET_ERR_DEVICE", 6: "JET_ERR_WORKSPACE",
          7: "JET_ERR_TIMEOUT"}
OP = {"quant_act_1x128": 0, "quant_w_128x128": 1, "requant_128x1": 2,
      "gemm_fp8_fwd": 3, "gemm_fp8_dgrad": 4, "gemm_fp8_wgrad": 5,
      "token_mult_prob_error": 6, "quant_dual_1x128_128x1": 7, "token_mismatch_masked": 8,
      "swiglu_quant_1x128": 9, "kv_calibrate": 10, "kv_cache_write": 11,
      "token_mismatch_per_sequence": 12, "rmsnorm_quant_1x128": 13}

# name -> argtypes (restype is int status unless listed in _RESTYPE)
P, I, Z = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
SIGNATURES = {
    "jet_status_str": [ctypes.c_int],
    "jet_version": [],
    "jet_quant_act_1x128": [P, I, I, P, P, P],
    "jet_quant_w_128x128": [P, I, I, P, P, P],
    "jet_requant_128x1": [P, P, I, I, P, P, P],
    "jet_quant_dual_1x128_128x1": [P, I, I, P, P, P, P, P],
    "jet_swiglu_quant_1x128": [P, P, I, I, I, P, P, P],
    "jet_rmsnorm_quant_1x128": [P, P, I, I, ctypes.c_float, P, P, P],
    "jet_kv_calibrate": [P, I, I, I, P, P],
    "jet_token_mismatch_per_sequence": [P, P, P, P, I, I, ctypes.c_float, P, P, P, P],
    "jet_kv_cache_write": [P, P, P, I, I, I, P, I, P],
    "jet_gemm_fp8_fwd": [P, P, P, P, I, I, I, P, P, Z, P],
    "jet_gemm_fp8_fwd_grouped": [P, P, P, P, P, I, I, I, I, P, P],
    "jet_gemm_fp8_dgrad_grouped": [P, P, P, P, P, I, I, I, I, P, P],
    "jet_gemm_fp8_wgrad_grouped": [P, P, P, P, P, I, I, I, I, P, P],
    "jet_gemm_fp8_dgrad": [P, P, P, P, I, I, I, P, P, Z, P],
    "jet_gemm_fp8_wgrad": [P, P, P, P, I, I, I, P, P, Z, P],
    "jet_token_mult_prob_error": [P, P, I, P, P, Z, P],
    "jet_token_mult_prob_error_noalloc": [P, P, I, P, P],
    "jet_token_mismatch_masked": [P, P, P, I, ctypes.c_float, P, P, P, P, Z, P],
    "jet_workspace_bytes": [ctypes.c_int, I, I, I],
    "jet_device_status": [P, ctypes.POINTER(ctypes.c_uint32)],
    "jet_selftest_bounded_wait": [ctypes.c_uint32, P],
    "jet_selftest_gemm_timeout": [P, P, P, P, I, I, I, P, ctypes.c_uint64, P],
    "jet_selftest_quotient": [P, P, I, P, P],
}
_RESTYPE = {"jet_status_str": ctypes.c_char_p, "jet_version": ctypes.c_int,
            "jet_workspace_bytes": ctypes.c_size_t}


class JetError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load (building first if needed) ``libjetfp8.so``; raises if impossible."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing and not _build.up_to_date():
            path = _build.build()
        if not os.path.exists(path):
            raise ImportError(f"jet_fp8 library not built: {path}")
        lib = ctypes.CDLL(path)
        for name, args in SIGNATURES.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = _RESTYPE.get(name, ctypes.c_int)
        _lib = lib
        return lib


def _check(fn: str, code: int):
    if code != 0:
        raise JetError(fn, code)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() > 0 else ctypes.c_void_p(0)


def _need(t, dtype, shape, name):
    import torch
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.numel() and (not t.is_cuda or not t.is_contiguous()):
        raise ValueError(f"{name}: must be a contiguous CUDA tensor")
    return t


def workspace_bytes(op: str, M=0, N=0, K=0) -> int:
    return int(load().jet_workspace_bytes(OP[op], M, N, K))


def selftest_bounded_wait(limit_us: int, stream=None):
    """Run the library's bounded-wait self-test kernel (records a timeout)."""
    _check("jet_selftest_bounded_wait", load().jet_selftest_bounded_wait(limit_us, _stream(stream)))


def selftest_gemm_timeout(qx, sx, qw, sw, limit_cycles: int, stream=None):
    """The forward product on the single-CTA GEMM kernel with its pipeline
    waits limited to `limit_cycles` SM cycles (the GEMM's time-out path);
    returns Y (unspecified when a wait ran out; see device_status())."""
    import torch
    M, K = qx.shape
    N = qw.shape[0]
    _need(qx, torch.uint8, (M, K), "qx")
    _need(sx, torch.float32, (K // 128, M), "sx")
    _need(qw, torch.uint8, (N, K), "qw")
    _need(sw, torch.float32, (N // 128, K // 128), "sw")
    y = torch.empty((M, N), dtype=torch.bfloat16, device=qx.device)
    _check("jet_selftest_gemm_timeout", load().jet_selftest_gemm_timeout(
        _ptr(qx), _ptr(sx), _ptr(qw), _ptr(sw), M, N, K, _ptr(y), limit_cycles, _stream(stream)))
    return y


def selftest_quotient(x, s, stream=None):
    """x / s elementwise through the quantizers' division routine."""
    import torch
    n = x.numel()
    _need(x, torch.float32, (n,), "x")
    _need(s, torch.float32, (n,), "s")
    q = torch.empty_like(x)
    _check("jet_selftest_quotient", load().jet_selftest_quotient(_ptr(x), _ptr(s), n, _ptr(q),
                                                                  _stream(stream)))
    return q


def device_status(stream=None):
    """(status code, raw status word) after synchronizing the stream."""
    detail = ctypes.c_uint32(0)
    code = load().jet_device_status(_stream(stream), ctypes.byref(detail))
    return code, detail.value


# --------------------------------------------------------------------------
# Entry points with the C names; tensors in, outputs written in place.
# --------------------------------------------------------------------------

def jet_quant_act_1x128(x, q, s, stream=None):
    import torch
    M, K = x.shape
    _need(x, torch.bfloat16, (M, K), "x")
    _need(q, torch.uint8, (M, K), "q")
    _need(s, torch.float32, (K // 128, M), "s")
    _check("jet_quant_act_1x128", load().jet_quant_act_1x128(
        _ptr(x), M, K, _ptr(q), _ptr(s), _stream(stream)))


def jet_quant_w_128x128(w, q, s, stream=None):
    import torch
    N, K = w.shape
    _need(w, torch.bfloat16, (N, K), "w")
    _need(q, torch.uint8, (N, K), "q")
    _need(s, torch.float32, (N // 128, K // 128), "s")
    _check("jet_quant_w_128x128", load().jet_quant_w_128x128(
        _ptr(w), N, K, _ptr(q), _ptr(s), _stream(stream)))


def jet_requant_128x1(q, s, qT, sT, stream=None):
    import torch
    M, K = q.shape
    _need(q, torch.uint8, (M, K), "q")
    _need(s, torch.float32, (K // 128, M), "s")
    _need(qT, torch.uint8, (K, M), "qT")
    _need(sT, torch.float32, (M // 128, K), "sT")
    _check("jet_requant_128x1", load().jet_requant_128x1(
        _ptr(q), _ptr(s), M, K, _ptr(qT), _ptr(sT), _stream(stream)))


def jet_quant_dual_1x128_128x1(x, q, s, qT, sT, stream=None):
    import torch
    M, K = x.shape
    _need(x, torch.bfloat16, (M, K), "x")
    _need(q, torch.uint8, (M, K), "q")
    _need(s, torch.float32, (K // 128, M), "s")
    _need(qT, torch.uint8, (K, M), "qT")
    _need(sT, torch.float32, (M // 128, K), "sT")
    _check("jet_quant_dual_1x128_128x1", load().jet_quant_dual_1x128_128x1(
        _ptr(x), M, K, _ptr(q), _ptr(s), _ptr(qT), _ptr(sT), _stream(stream)))


def jet_swiglu_quant_1x128(gate, up, q, s, stream=None):
    """gate, up: [M, F] BF16 views whose rows may be strided (e.g. the two
    halves of a [M, 2F] gate_up product); both must share the row stride."""
    import torch
    M, F = gate.shape
    for t, name in ((gate, "gate"), (up, "up")):
        if t.dtype != torch.bfloat16 or tuple(t.shape) != (M, F):
            raise ValueError(f"{name}: expected bfloat16 [{M}, {F}]")
        if t.numel() and (not t.is_cuda or t.stride(1) != 1):
            raise ValueError(f"{name}: must be a CUDA tensor with contiguous rows")
    ld = gate.stride(0) if M > 1 else F
    if M > 1 and up.stride(0) != ld:
        raise ValueError("gate and up must have the same row stride")
    _need(q, torch.uint8, (M, F), "q")
    _need(s, torch.float32, (F // 128, M), "s")
    _check("jet_swiglu_quant_1x128", load().jet_swiglu_quant_1x128(
        _ptr(gate), _ptr(up), ld, M, F, _ptr(q), _ptr(s), _stream(stream)))


def jet_rmsnorm_quant_1x128(x, g, eps, q, s, stream=None):
    import torch
    M, K = x.shape
    _need(x, torch.bfloat16, (M, K), "x")
    _need(g, torch.bfloat16, (K,), "g")
    _need(q, torch.uint8, (M, K), "q")
    _need(s, torch.float32, (K // 128, M), "s")
    _check("jet_rmsnorm_quant_1x128", load().jet_rmsnorm_quant_1x128(
        _ptr(x), _ptr(g), M, K, float(eps), _ptr(q), _ptr(s), _stream(stream)))


def jet_kv_calibrate(x, scale, stream=None):
    """Per-head scales of the calibration batch x [T, H, D] (BF16) into scale [H]."""
    import torch
    T, H, D = x.shape
    _need(x, torch.bfloat16, (T, H, D), "x")
    _need(scale, torch.float32, (H,), "scale")
    _check("jet_kv_calibrate", load().jet_kv_calibrate(_ptr(x), T, H, D, _ptr(scale),
                                                       _stream(stream)))


def jet_kv_cache_write(x, scale, slots, cache, stream=None):
    """Write x [T, H, D] (BF16) as E4M3 codes into cache [S, H, D] at rows slots [T]."""
    import torch
    T, H, D = x.shape
    S = cache.shape[0]
    _need(x, torch.bfloat16, (T, H, D), "x")
    _need(scale, torch.float32, (H,), "scale")
    _need(slots, torch.int64, (T,), "slots")
    _need(cache, torch.uint8, (S, H, D), "cache")
    _check("jet_kv_cache_write", load().jet_kv_cache_write(
        _ptr(x), _ptr(scale), _ptr(slots), T, H, D, _ptr(cache), S, _stream(stream)))


def jet_token_mismatch_per_sequence(logp_train, logp_rollout, mask, seq_offsets, cap, w, out,
                                    count, stream=None):
    """Per-sequence mismatch metric and importance weights (see the header)."""
    import torch
    n = logp_train.numel()
    S = seq_offsets.numel() - 1
    _need(logp_train, torch.float32, (n,), "logp_train")
    _need(logp_rollout, torch.float32, (n,), "logp_rollout")
    if mask is not None:
        _need(mask, torch.uint8, (n,), "mask")
    _need(seq_offsets, torch.int64, (S + 1,), "seq_offsets")
    if w is not None:
        _need(w, torch.float32, (n,), "w")
    _need(out, torch.float32, (S,), "out")
    if count is not None:
        _need(count, torch.int64, (S,), "count")
    _check("jet_token_mismatch_per_sequence", load().jet_token_mismatch_per_sequence(
        _ptr(logp_train), _ptr(logp_rollout), _ptr(mask), _ptr(seq_offsets), S, n,
        float(cap), _ptr(w), _ptr(out), _ptr(count), _stream(stream)))


def token_mismatch_per_sequence(logp_train, logp_rollout, seq_offsets, mask=None, cap=0.0,
                                stream=None):
    """(metric [S], count [S], w [n]) on the device."""
    import torch
    n, S, dev = logp_train.numel(), seq_offsets.numel() - 1, logp_train.device
    out = torch.empty((S,), dtype=torch.float32, device=dev)
    count = torch.empty((S,), dtype=torch.int64, device=dev)
    w = torch.empty((n,), dtype=torch.float32, device=dev)
    jet_token_mismatch_per_sequence(logp_train, logp_rollout, mask, seq_offsets, cap, w, out,
                                    count, stream)
    return out, count, w


def kv_calibrate(x, stream=None):
    """scale [H] FP32 of the calibration batch x [T, H, D]."""
    import torch
    scale = torch.empty((x.shape[1],), dtype=torch.float32, device=x.device)
    jet_kv_calibrate(x, scale, stream)
    return scale


def _gemm(name, a, sa, b, sb, M, N, K, out, ws, stream):
    if ws is None:  # the split-contraction partials of small-M products
        ws = _ws(name[4:], M, N, K, out.device)
    ws_ptr, ws_bytes = (_ptr(ws), ws.numel() * ws.element_size()) if ws is not None else (ctypes.c_void_p(0), 0)
    _check(name, getattr(load(), name)(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), M, N, K,
                                       _ptr(out), ws_ptr, ws_bytes, _stream(stream)))


def jet_gemm_fp8_fwd(qx, sx, qw, sw, y, ws=None, stream=None):
    import torch
    M, K = qx.shape
    N = qw.shape[0]
    _need(qx, torch.uint8, (M, K), "qx")
    _need(sx, torch.float32, (K // 128, M), "sx")
    _need(qw, torch.uint8, (N, K), "qw")
    _need(sw, torch.float32, (N // 128, K // 128), "sw")
    _need(y, torch.bfloat16, (M, N), "y")
    _gemm("jet_gemm_fp8_fwd", qx, sx, qw, sw, M, N, K, y, ws, stream)


def jet_gemm_fp8_fwd_grouped(qx, sx, qw, sw, offsets, y, stream=None):
    """Expert-grouped forward product; ``offsets`` is the int64 device tensor
    of the E+1 row offsets of the experts' tokens in ``qx``."""
    import torch
    M, K = qx.shape
    E, N = qw.shape[0], qw.shape[1]
    _need(qx, torch.uint8, (M, K), "qx")
    _need(sx, torch.float32, (K // 128, M), "sx")
    _need(qw, torch.uint8, (E, N, K), "qw")
    _need(sw, torch.float32, (E, N // 128, K // 128), "sw")
    _need(offsets, torch.int64, (E + 1,), "offsets")
    _need(y, torch.bfloat16, (M, N), "y")
    _check("jet_gemm_fp8_fwd_grouped", load().jet_gemm_fp8_fwd_grouped(
        _ptr(qx), _ptr(sx), _ptr(qw), _ptr(sw), _ptr(offsets), E, M, N, K, _ptr(y),
        _stream(stream)))


def jet_gemm_fp8_dgrad_grouped(qdy, sdy, qw, sw, offsets, dx, stream=None):
    """Expert-grouped DGrad; ``offsets`` as in jet_gemm_fp8_fwd_grouped."""
    import torch
    M, N = qdy.shape
    E, K = qw.shape[0], qw.shape[2]
    _need(qdy, torch.uint8, (M, N), "qdy")
    _need(sdy, torch.float32, (N // 128, M), "sdy")
    _need(qw, torch.uint8, (E, N, K), "qw")
    _need(sw, torch.float32, (E, N // 128, K // 128), "sw")
    _need(offsets, torch.int64, (E + 1,), "offsets")
    _need(dx, torch.bfloat16, (M, K), "dx")
    _check("jet_gemm_fp8_dgrad_grouped", load().jet_gemm_fp8_dgrad_grouped(
        _ptr(qdy), _ptr(sdy), _ptr(qw), _ptr(sw), _ptr(offsets), E, M, N, K, _ptr(dx),
        _stream(stream)))


def jet_gemm_fp8_wgrad_grouped(qdyT, sdyT, qxT, sxT, offsets, dw, stream=None):
    """Expert-grouped WGrad over each expert's tokens; offsets in multiples of 128."""
    import torch
    N, M = qdyT.shape
    K = qxT.shape[0]
    E = offsets.shape[0] - 1
    _need(qdyT, torch.uint8, (N, M), "qdyT")
    _need(sdyT, torch.float32, (M // 128, N), "sdyT")
    _need(qxT, torch.uint8, (K, M), "qxT")
    _need(sxT, torch.float32, (M // 128, K), "sxT")
    _need(offsets, torch.int64, (E + 1,), "offsets")
    _need(dw, torch.bfloat16, (E, N, K), "dw")
    _check("jet_gemm_fp8_wgrad_grouped", load().jet_gemm_fp8_wgrad_grouped(
        _ptr(qdyT), _ptr(sdyT), _ptr(qxT), _ptr(sxT), _ptr(offsets), E, M, N, K, _ptr(dw),
        _stream(stream)))


def jet_gemm_fp8_dgrad(qdy, sdy, qw, sw, dx, ws=None, stream=None):
    import torch
    M, N = qdy.shape
    K = qw.shape[1]
    _need(qdy, torch.uint8, (M, N), "qdy")
    _need(sdy, torch.float32, (N // 128, M), "sdy")
    _need(qw, torch.uint8, (N, K), "qw")
    _need(sw, torch.float32, (N // 128, K // 128), "sw")
    _need(dx, torch.bfloat16, (M, K), "dx")
    _gemm("jet_gemm_fp8_dgrad", qdy, sdy, qw, sw, M, N, K, dx, ws, stream)


def jet_gemm_fp8_wgrad(qdyT, sdyT, qxT, sxT, dw, ws=None, stream=None):
    import torch
    N, M = qdyT.shape
    K = qxT.shape[0]
    _need(qdyT, torch.uint8, (N, M), "qdyT")
    _need(sdyT, torch.float32, (M // 128, N), "sdyT")
    _need(qxT, torch.uint8, (K, M), "qxT")
    _need(sxT, torch.float32, (M // 128, K), "sxT")
    _need(dw, torch.bfloat16, (N, K), "dw")
    _gemm("jet_gemm_fp8_wgrad", qdyT, sdyT, qxT, sxT, M, N, K, dw, ws, stream)


def jet_token_mult_prob_error(logp_train, logp_rollout, out, ws, stream=None):
    import torch
    n = logp_train.numel()
    _need(logp_train, torch.float32, (n,), "logp_train")
    _need(logp_rollout, torch.float32, (n,), "logp_rollout")
    _need(out, torch.float32, (1,), "out")
    _check("jet_token_mult_prob_error", load().jet_token_mult_prob_error(
        _ptr(logp_train), _ptr(logp_rollout), n, _ptr(out), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def jet_token_mult_prob_error_noalloc(logp_train, logp_rollout, out, stream=None):
    """Same metric with the library's static scratch instead of a workspace."""
    import torch
    n = logp_train.numel()
    _need(logp_train, torch.float32, (n,), "logp_train")
    _need(logp_rollout, torch.float32, (n,), "logp_rollout")
    _need(out, torch.float32, (1,), "out")
    _check("jet_token_mult_prob_error_noalloc", load().jet_token_mult_prob_error_noalloc(
        _ptr(logp_train), _ptr(logp_rollout), n, _ptr(out), _stream(stream)))


def jet_token_mismatch_masked(logp_train, logp_rollout, mask, cap, w, out, count, ws,
                              stream=None):
    import torch
    n = logp_train.numel()
    _need(logp_train, torch.float32, (n,), "logp_train")
    _need(logp_rollout, torch.float32, (n,), "logp_rollout")
    if mask is not None:
        _need(mask, torch.uint8, (n,), "mask")
    if w is not None:
        _need(w, torch.float32, (n,), "w")
    _need(out, torch.float32, (1,), "out")
    if count is not None:
        _need(count, torch.int64, (1,), "count")
    _check("jet_token_mismatch_masked", load().jet_token_mismatch_masked(
        _ptr(logp_train), _ptr(logp_rollout), _ptr(mask), n, float(cap), _ptr(w), _ptr(out),
        _ptr(count), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


# --------------------------------------------------------------------------
# Allocation helpers (torch owns the memory; the library never allocates).
# --------------------------------------------------------------------------

def quant_act_1x128(x, stream=None):
    import torch
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    s = torch.empty((K // 128, M), dtype=torch.float32, device=x.device)
    jet_quant_act_1x128(x, q, s, stream)
    return q, s


def quant_w_128x128(w, stream=None):
    import torch
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    s = torch.empty((N // 128, K // 128), dtype=torch.float32, device=w.device)
    jet_quant_w_128x128(w, q, s, stream)
    return q, s


def requant_128x1(q, s, stream=None):
    import torch
    M, K = q.shape
    qT = torch.empty((K, M), dtype=torch.uint8, device=q.device)
    sT = torch.empty((M // 128, K), dtype=torch.float32, device=q.device)
    jet_requant_128x1(q, s, qT, sT, stream)
    return qT, sT


def quant_dual_1x128_128x1(x, stream=None):
    """(q, s, qT, sT): the 1x128 and the transposed 128x1 forms of x."""
    import torch
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    s = torch.empty((K // 128, M), dtype=torch.float32, device=x.device)
    qT = torch.empty((K, M), dtype=torch.uint8, device=x.device)
    sT = torch.empty((M // 128, K), dtype=torch.float32, device=x.device)
    jet_quant_dual_1x128_128x1(x, q, s, qT, sT, stream)
    return q, s, qT, sT


def rmsnorm_quant_1x128(x, g, eps=1e-5, stream=None):
    """RMSNorm of x [M,K] with gain g [K] fused with the 1x128 quantization:
    (codes uint8 [M,K], scales float32 [K/128, M])."""
    import torch
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    s = torch.empty((K // 128, M), dtype=torch.float32, device=x.device)
    jet_rmsnorm_quant_1x128(x, g, eps, q, s, stream)
    return q, s


def swiglu_quant_1x128(gate, up, stream=None):
    """(q, s): the 1x128 form of silu(gate) * up."""
    import torch
    M, F = gate.shape
    q = torch.empty((M, F), dtype=torch.uint8, device=gate.device)
    s = torch.empty((F // 128, M), dtype=torch.float32, device=gate.device)
    jet_swiglu_quant_1x128(gate, up, q, s, stream)
    return q, s


def _ws(op, M, N, K, device):
    import torch
    nb = workspace_bytes(op, M, N, K)
    return torch.empty((max(nb, 16),), dtype=torch.uint8, device=device) if nb else None


def gemm_fp8_fwd(qx, sx, qw, sw, stream=None):
    import torch
    M, K = qx.shape
    N = qw.shape[0]
    y = torch.empty((M, N), dtype=torch.bfloat16, device=qx.device)
    jet_gemm_fp8_fwd(qx, sx, qw, sw, y, _ws("gemm_fp8_fwd", M, N, K, qx.device), stream)
    return y


def gemm_fp8_fwd_grouped(qx, sx, qw, sw, offsets, stream=None):
    """Y [M][N] BF16: every expert's tokens times that expert's weights."""
    import torch
    M, N = qx.shape[0], qw.shape[1]
    y = torch.empty((M, N), dtype=torch.bfloat16, device=qx.device)
    jet_gemm_fp8_fwd_grouped(qx, sx, qw, sw, offsets, y, stream)
    return y


def gemm_fp8_dgrad_grouped(qdy, sdy, qw, sw, offsets, stream=None):
    """dX [M][K] BF16: every expert's token rows times that expert's weights."""
    import torch
    M, K = qdy.shape[0], qw.shape[2]
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=qdy.device)
    jet_gemm_fp8_dgrad_grouped(qdy, sdy, qw, sw, offsets, dx, stream)
    return dx


def gemm_fp8_wgrad_grouped(qdyT, sdyT, qxT, sxT, offsets, stream=None):
    """dW [E][N][K] BF16: every expert's weight gradient over its own tokens."""
    import torch
    N, K, E = qdyT.shape[0], qxT.shape[0], offsets.shape[0] - 1
    dw = torch.empty((E, N, K), dtype=torch.bfloat16, device=qdyT.device)
    jet_gemm_fp8_wgrad_grouped(qdyT, sdyT, qxT, sxT, offsets, dw, stream)
    return dw


def gemm_fp8_dgrad(qdy, sdy, qw, sw, stream=None):
    import torch
    M, N = qdy.shape
    K = qw.shape[1]
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=qdy.device)
    jet_gemm_fp8_dgrad(qdy, sdy, qw, sw, dx, _ws("gemm_fp8_dgrad", M, N, K, qdy.device), stream)
    return dx


def gemm_fp8_wgrad(qdyT, sdyT, qxT, sxT, stream=None):
    import torch
    N, M = qdyT.shape
    K = qxT.shape[0]
    dw = torch.empty((N, K), dtype=torch.bfloat16, device=qdyT.device)
    jet_gemm_fp8_wgrad(qdyT, sdyT, qxT, sxT, dw, _ws("gemm_fp8_wgrad", M, N, K, qdyT.device), stream)
    return dw


def token_mult_prob_error(logp_train, logp_rollout, stream=None):
    import torch
    n = logp_train.numel()
    out = torch.empty((1,), dtype=torch.float32, device=logp_train.device)
    ws = torch.empty((max(workspace_bytes("token_mult_prob_error", n), 16),),
                     dtype=torch.uint8, device=logp_train.device)
    jet_token_mult_prob_error(logp_train, logp_rollout, out, ws, stream)
    return out


def token_mismatch_masked(logp_train, logp_rollout, mask=None, cap: float = 0.0, stream=None):
    """(metric [1], count [1], w [n]) for the masked tokens; see the C header."""
    import torch
    n = logp_train.numel()
    dev = logp_train.device
    out = torch.empty((1,), dtype=torch.float32, device=dev)
    count = torch.empty((1,), dtype=torch.int64, device=dev)
    w = torch.empty((n,), dtype=torch.float32, device=dev)
    ws = torch.empty((max(workspace_bytes("token_mismatch_masked", n), 16),), dtype=torch.uint8,
                     device=dev)
    jet_token_mismatch_masked(logp_train, logp_rollout, mask, cap, w, out, count, ws, stream)
    return out, count, w
