"""The C-ABI library builds, loads and exports every symbol of include/jet_fp8.h,
and its host-side argument checks return the documented codes (CPU only: no
call here reaches a kernel launch)."""
import ctypes
import os
import re

import pytest

from fp8_block_quantized_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "jet_fp8.h")

OK, NULL, SHAPE, ALIGN, CUDA, DEVICE, WORKSPACE, TIMEOUT = range(8)
V = ctypes.c_void_p


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"JET_API\s+[\w\s\*]*?\b(jet_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return binding.load()


def fake(addr):
    """A non-dereferenced stand-in pointer (argument checks fail before any use)."""
    return V(addr)


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) >= set(binding.SIGNATURES)


def test_status_strings(lib):
    for code, name in binding.STATUS.items():
        assert lib.jet_status_str(code).decode() == name
    assert lib.jet_status_str(99).decode() == "JET_ERR_UNKNOWN"
    assert lib.jet_version() >= 10000


def test_workspace_bytes(lib):
    op = binding.OP
    for name in ("quant_act_1x128", "quant_w_128x128", "requant_128x1",
                 "gemm_fp8_fwd", "gemm_fp8_dgrad", "gemm_fp8_wgrad"):
        assert lib.jet_workspace_bytes(op[name], 8192, 4096, 4096) == 0
    # split contraction for at most 512 output rows: FP32 partials [splits][R][C];
    # about 128 units of 128-wide tiles (of 256-wide ones when that gives one),
    # at most 8 ranges per tile, partials at most 32 MB
    fwd, dgrad, wgrad = op["gemm_fp8_fwd"], op["gemm_fp8_dgrad"], op["gemm_fp8_wgrad"]
    assert lib.jet_workspace_bytes(fwd, 1, 4096, 4096) == 0                     # decode kernel
    assert lib.jet_workspace_bytes(fwd, 1, 14336, 4096) == 0                    # one token: always
    assert lib.jet_workspace_bytes(fwd, 2, 4096, 4096) == 0                     # M N K = 2^25
    assert lib.jet_workspace_bytes(fwd, 4, 1024, 4096) == 0
    assert lib.jet_workspace_bytes(fwd, 4, 4096, 4096) == 4 * 4 * 4096 * 4      # 32 tiles
    assert lib.jet_workspace_bytes(fwd, 2, 14336, 4096) == 2 * 2 * 14336 * 4    # 112: 56 of 256
    assert lib.jet_workspace_bytes(fwd, 5, 4096, 4096) == 4 * 5 * 4096 * 4
    assert lib.jet_workspace_bytes(fwd, 64, 4096, 4096) == 4 * 64 * 4096 * 4
    assert lib.jet_workspace_bytes(fwd, 64, 14336, 4096) == 2 * 64 * 14336 * 4
    assert lib.jet_workspace_bytes(fwd, 16, 1024, 4096) == 8 * 16 * 1024 * 4    # 8 tiles: at most 8
    assert lib.jet_workspace_bytes(fwd, 128, 128, 128) == 0                     # one slice
    assert lib.jet_workspace_bytes(fwd, 129, 4096, 4096) == 2 * 129 * 4096 * 4  # two row tiles
    assert lib.jet_workspace_bytes(fwd, 256, 4096, 14336) == 2 * 256 * 4096 * 4
    assert lib.jet_workspace_bytes(fwd, 513, 4096, 14336) == 0                  # pair kernel
    assert lib.jet_workspace_bytes(fwd, 256, 14336, 4096) == 0                  # 112 of 256
    assert lib.jet_workspace_bytes(fwd, 128, 4096, 1024) == 4 * 128 * 4096 * 4  # two slices each
    assert lib.jet_workspace_bytes(fwd, 512, 4096, 14336) == 2 * 512 * 4096 * 4  # 64 of 256
    assert lib.jet_workspace_bytes(fwd, 512, 8192, 4096) == 0                   # 128 of 256
    assert lib.jet_workspace_bytes(dgrad, 16, 4096, 1024) == 8 * 16 * 1024 * 4  # C = K = 1024
    assert lib.jet_workspace_bytes(dgrad, 16, 1024, 4096) == 4 * 16 * 4096 * 4
    assert lib.jet_workspace_bytes(wgrad, 128, 128, 4096) == 0
    m = op["token_mult_prob_error"]
    assert lib.jet_workspace_bytes(m, 1, 0, 0) == 8
    assert lib.jet_workspace_bytes(m, 2048, 0, 0) == 8
    assert lib.jet_workspace_bytes(m, 2049, 0, 0) == 16
    assert lib.jet_workspace_bytes(m, 4 * 1024 * 1024, 0, 0) == 1024 * 8
    assert lib.jet_workspace_bytes(m, 0, 0, 0) == 0
    assert lib.jet_workspace_bytes(m, -5, 0, 0) == 0
    assert lib.jet_workspace_bytes(42, 1, 1, 1) == 0


A = 0x10000  # 16-byte aligned stand-ins
B = 0x20000
C = 0x30000
D = 0x40000
MIS = 0x10008  # 8-byte aligned only


def test_quant_act_checks(lib):
    f = lib.jet_quant_act_1x128
    assert f(None, 4, 128, fake(B), fake(C), None) == NULL
    assert f(fake(A), 4, 128, None, fake(C), None) == NULL
    assert f(fake(A), 4, 128, fake(B), None, None) == NULL
    assert f(fake(A), -1, 128, fake(B), fake(C), None) == SHAPE
    assert f(fake(A), 4, 100, fake(B), fake(C), None) == SHAPE
    assert f(fake(MIS), 4, 128, fake(B), fake(C), None) == ALIGN
    assert f(fake(A), 4, 128, fake(B), fake(MIS), None) == ALIGN


def test_quant_dual_checks(lib):
    f = lib.jet_quant_dual_1x128_128x1
    ok = [fake(A), 128, 128, fake(B), fake(C), fake(D), fake(A + 0x1000)]
    assert f(None, *ok[1:], None) == NULL
    assert f(*ok[:6], None, None) == NULL
    assert f(ok[0], 100, 128, *ok[3:], None) == SHAPE       # tokens must hold whole 128x1 groups
    assert f(ok[0], 128, 100, *ok[3:], None) == SHAPE
    assert f(ok[0], -128, 128, *ok[3:], None) == SHAPE
    assert f(*ok[:5], fake(MIS), ok[6], None) == ALIGN
    assert f(None, 0, 128, None, None, None, None, None) in (OK, DEVICE)   # empty: nothing to do
    assert lib.jet_workspace_bytes(binding.OP["quant_dual_1x128_128x1"], 8192, 4096, 0) == 0


def test_quant_w_and_requant_checks(lib):
    w = lib.jet_quant_w_128x128
    assert w(None, 128, 128, fake(B), fake(C), None) == NULL
    assert w(fake(A), 100, 128, fake(B), fake(C), None) == SHAPE
    assert w(fake(A), 128, 129, fake(B), fake(C), None) == SHAPE
    assert w(fake(A), 128, 128, fake(MIS), fake(C), None) == ALIGN
    r = lib.jet_requant_128x1
    assert r(fake(A), None, 128, 128, fake(C), fake(D), None) == NULL
    assert r(fake(A), fake(B), 100, 128, fake(C), fake(D), None) == SHAPE   # M % 128
    assert r(fake(A), fake(B), 128, 100, fake(C), fake(D), None) == SHAPE
    assert r(fake(A), fake(B), 128, 128, fake(C), fake(MIS), None) == ALIGN


@pytest.mark.parametrize("name", ["jet_gemm_fp8_fwd", "jet_gemm_fp8_dgrad", "jet_gemm_fp8_wgrad"])
def test_gemm_checks(lib, name):
    f = getattr(lib, name)
    args = [fake(A), fake(B), fake(C), fake(D)]
    assert f(*args, 128, 128, 128, None, None, 0, None) == NULL          # no output
    assert f(None, fake(B), fake(C), fake(D), 128, 128, 128, fake(A), None, 0, None) == NULL
    assert f(*args, -1, 128, 128, fake(A), None, 0, None) == SHAPE
    assert f(*args, 128, 100, 128, fake(A), None, 0, None) == SHAPE
    assert f(*args, 128, 128, 100, fake(A), None, 0, None) == SHAPE
    assert f(*args, 128, 128, 128, fake(MIS), None, 0, None) == ALIGN
    assert f(fake(MIS), fake(B), fake(C), fake(D), 128, 128, 128, fake(A), None, 0, None) == ALIGN
    if name == "jet_gemm_fp8_wgrad":      # the token axis must hold whole 128-groups
        assert f(*args, 100, 128, 128, fake(A), None, 0, None) == SHAPE
    else:                                 # a split small-M product needs its partials
        need = lib.jet_workspace_bytes(binding.OP[name[4:]], 16, 1024, 1024)
        assert need > 0
        assert f(*args, 16, 1024, 1024, fake(A), None, 0, None) == WORKSPACE
        assert f(*args, 16, 1024, 1024, fake(A), fake(B), need - 16, None) == WORKSPACE
        assert f(*args, 16, 1024, 1024, fake(A), fake(MIS), need, None) == ALIGN


def test_swiglu_quant_checks(lib):
    f = lib.jet_swiglu_quant_1x128
    assert f(None, fake(B), 256, 4, 256, fake(C), fake(D), None) == NULL
    assert f(fake(A), fake(B), 256, 4, 256, fake(C), None, None) == NULL
    assert f(fake(A), fake(B), 256, -1, 256, fake(C), fake(D), None) == SHAPE
    assert f(fake(A), fake(B), 256, 4, 200, fake(C), fake(D), None) == SHAPE   # F % 128
    assert f(fake(A), fake(B), 128, 4, 256, fake(C), fake(D), None) == SHAPE   # ld < F
    assert f(fake(A), fake(B), 260, 4, 256, fake(C), fake(D), None) == ALIGN   # rows not 16 B apart
    assert f(fake(MIS), fake(B), 256, 4, 256, fake(C), fake(D), None) == ALIGN
    assert f(fake(A), fake(MIS), 512, 4, 256, fake(C), fake(D), None) == ALIGN
    assert lib.jet_workspace_bytes(binding.OP["swiglu_quant_1x128"], 4, 0, 256) == 0


def test_rmsnorm_quant_checks(lib):
    f = lib.jet_rmsnorm_quant_1x128
    assert f(None, fake(B), 4, 256, 1e-5, fake(C), fake(D), None) == NULL
    assert f(fake(A), None, 4, 256, 1e-5, fake(C), fake(D), None) == NULL
    assert f(fake(A), fake(B), 4, 256, 1e-5, fake(C), None, None) == NULL
    assert f(fake(A), fake(B), -1, 256, 1e-5, fake(C), fake(D), None) == SHAPE
    assert f(fake(A), fake(B), 4, 200, 1e-5, fake(C), fake(D), None) == SHAPE     # K % 128
    assert f(fake(A), fake(B), 4, 256, -1.0, fake(C), fake(D), None) == SHAPE     # eps < 0
    assert f(fake(A), fake(B), 4, 256, float("nan"), fake(C), fake(D), None) == SHAPE
    assert f(fake(A), fake(B), 4, 256, float("inf"), fake(C), fake(D), None) == SHAPE
    assert f(fake(MIS), fake(B), 4, 256, 1e-5, fake(C), fake(D), None) == ALIGN
    assert f(fake(A), fake(MIS), 4, 256, 1e-5, fake(C), fake(D), None) == ALIGN
    assert f(None, None, 0, 256, 1e-5, None, None, None) in (OK, DEVICE)        # empty
    assert lib.jet_workspace_bytes(binding.OP["rmsnorm_quant_1x128"], 4, 0, 256) == 0


def test_grouped_gemm_checks(lib):
    f = lib.jet_gemm_fp8_fwd_grouped
    args = [fake(A), fake(B), fake(C), fake(D)]
    assert f(*args, fake(A), 8, 256, 128, 128, None, None) == NULL        # no output
    assert f(*args, None, 8, 256, 128, 128, fake(A), None) == NULL        # no offsets
    assert f(None, fake(B), fake(C), fake(D), fake(A), 8, 256, 128, 128, fake(A), None) == NULL
    assert f(*args, fake(A), 0, 256, 128, 128, fake(A), None) == SHAPE    # no expert
    assert f(*args, fake(A), 385, 256, 128, 128, fake(A), None) == SHAPE  # over the limit
    assert f(*args, fake(A), 8, -1, 128, 128, fake(A), None) == SHAPE
    assert f(*args, fake(A), 8, 256, 100, 128, fake(A), None) == SHAPE
    assert f(*args, fake(A), 8, 256, 128, 100, fake(A), None) == SHAPE
    assert f(*args, fake(A), 384, 256, 1 << 22, 128, fake(A), None) == SHAPE  # E*N rows
    assert f(*args, fake(MIS), 8, 256, 128, 128, fake(A), None) == ALIGN
    assert f(*args, fake(A), 8, 256, 128, 128, fake(MIS), None) == ALIGN
    # an empty output needs no pointer at all; empty experts are no error
    assert f(None, None, None, None, None, 8, 0, 128, 128, None, None) in (OK, DEVICE)


@pytest.mark.parametrize("name", ["jet_gemm_fp8_dgrad_grouped", "jet_gemm_fp8_wgrad_grouped"])
def test_grouped_backward_checks(lib, name):
    f = getattr(lib, name)
    args = [fake(A), fake(B), fake(C), fake(D)]
    assert f(*args, fake(A), 8, 256, 128, 128, None, None) == NULL
    assert f(*args, None, 8, 256, 128, 128, fake(A), None) == NULL
    assert f(*args, fake(A), 0, 256, 128, 128, fake(A), None) == SHAPE
    assert f(*args, fake(A), 385, 256, 128, 128, fake(A), None) == SHAPE
    assert f(*args, fake(A), 8, 256, 100, 128, fake(A), None) == SHAPE
    assert f(*args, fake(A), 8, 256, 128, 100, fake(A), None) == SHAPE
    assert f(*args, fake(MIS), 8, 256, 128, 128, fake(A), None) == ALIGN
    assert f(*args, fake(A), 8, 256, 128, 128, fake(MIS), None) == ALIGN
    if name == "jet_gemm_fp8_wgrad_grouped":   # tokens are the 128x1 group axis
        assert f(*args, fake(A), 8, 200, 128, 128, fake(A), None) == SHAPE


def test_kv_cache_checks(lib):
    cal, wr = lib.jet_kv_calibrate, lib.jet_kv_cache_write
    assert cal(fake(A), 4, 8, 100, fake(B), None) == SHAPE       # D % 16
    assert cal(fake(A), 4, 1025, 128, fake(B), None) == SHAPE    # too many heads
    assert cal(fake(A), -1, 8, 128, fake(B), None) == SHAPE
    assert cal(None, 4, 8, 128, fake(B), None) == NULL
    assert cal(fake(A), 4, 8, 128, None, None) == NULL
    assert cal(fake(MIS), 4, 8, 128, fake(B), None) == ALIGN
    assert wr(fake(A), fake(B), fake(C), 4, 8, 128, None, 16, None) == NULL
    assert wr(fake(A), fake(B), None, 4, 8, 128, fake(D), 16, None) == NULL
    assert wr(fake(A), fake(B), fake(C), 4, 8, 128, fake(D), -1, None) == SHAPE
    assert wr(fake(A), fake(B), fake(MIS), 4, 8, 128, fake(D), 16, None) == ALIGN
    assert lib.jet_workspace_bytes(binding.OP["kv_cache_write"], 4, 8, 128) == 0


def test_size_limits(lib):
    """Sizes past the documented limits are refused before anything runs."""
    big = 1 << 31
    assert lib.jet_quant_act_1x128(fake(A), big, 128, fake(B), fake(C), None) == SHAPE
    assert lib.jet_quant_w_128x128(fake(A), 128, big, fake(B), fake(C), None) == SHAPE
    g = lib.jet_gemm_fp8_fwd
    assert g(fake(A), fake(B), fake(C), fake(D), 1 << 30, 128, 128, fake(A), None, 0, None) == SHAPE
    assert g(fake(A), fake(B), fake(C), fake(D), 128, 1 << 30, 128, fake(A), None, 0, None) == SHAPE
    assert lib.jet_swiglu_quant_1x128(fake(A), fake(B), 256, big, 256, fake(C), fake(D),
                                      None) == SHAPE
    assert lib.jet_kv_cache_write(fake(A), fake(B), fake(C), 4, 1024, 1 << 20, fake(D), 16,
                                  None) == SHAPE


def test_per_sequence_metric_checks(lib):
    f = lib.jet_token_mismatch_per_sequence
    assert f(fake(A), fake(B), None, None, 4, 16, 0.0, None, fake(C), None, None) == NULL
    assert f(fake(A), fake(B), None, fake(D), 4, 16, 0.0, None, None, None, None) == NULL
    assert f(None, fake(B), None, fake(D), 4, 16, 0.0, None, fake(C), None, None) == NULL
    assert f(fake(A), fake(B), None, fake(D), 0, 16, 0.0, None, fake(C), None, None) == SHAPE
    assert f(fake(A), fake(B), None, fake(D), 4, -1, 0.0, None, fake(C), None, None) == SHAPE
    assert f(fake(A), fake(B), fake(MIS), fake(D), 4, 16, 0.0, None, fake(C), None, None) == ALIGN


def test_metric_checks(lib):
    f = lib.jet_token_mult_prob_error
    assert f(None, fake(B), 16, fake(C), fake(D), 8, None) == NULL
    assert f(fake(A), fake(B), 0, fake(C), fake(D), 8, None) == SHAPE
    assert f(fake(A), fake(B), 16, fake(MIS), fake(D), 8, None) == ALIGN
    assert f(fake(A), fake(B), 16, fake(C), None, 0, None) == WORKSPACE
    assert f(fake(A), fake(B), 4096, fake(C), fake(D), 8, None) == WORKSPACE  # needs 16


def test_masked_metric_checks(lib):
    f = lib.jet_token_mismatch_masked
    op = binding.OP["token_mismatch_masked"]
    need = lib.jet_workspace_bytes(op, 4096, 0, 0)
    assert need == 2 * 8 * 2                               # two blocks: a sum and a count each
    assert f(None, fake(B), None, 16, 0.0, None, fake(C), None, fake(D), 64, None) == NULL
    assert f(fake(A), fake(B), None, 16, 0.0, None, None, None, fake(D), 64, None) == NULL
    assert f(fake(A), fake(B), None, 0, 0.0, None, fake(C), None, fake(D), 64, None) == SHAPE
    assert f(fake(A), fake(B), fake(MIS), 16, 0.0, None, fake(C), None, fake(D), 64, None) == ALIGN
    assert f(fake(A), fake(B), None, 16, 0.0, None, fake(C), None, None, 0, None) == WORKSPACE
    assert f(fake(A), fake(B), None, 4096, 0.0, None, fake(C), None, fake(D), need - 8, None) == WORKSPACE


def test_selftest_limit_checks(lib):
    assert lib.jet_selftest_bounded_wait(0, None) == SHAPE
    assert lib.jet_selftest_bounded_wait(2_000_000, None) == SHAPE
    f = lib.jet_selftest_gemm_timeout
    args = (fake(A), fake(B), fake(C), fake(D))
    assert f(None, fake(B), fake(C), fake(D), 128, 256, 256, fake(A), 100, None) == NULL
    assert f(*args, 129, 256, 256, fake(A), 100, None) == SHAPE       # at most 128 rows
    assert f(*args, 0, 256, 256, fake(A), 100, None) == SHAPE
    assert f(*args, 128, 200, 256, fake(A), 100, None) == SHAPE
    assert f(*args, 128, 256, 256, fake(A), 0, None) == SHAPE         # limit out of range
    assert f(*args, 128, 256, 256, fake(A), 4_000_000_001, None) == SHAPE
    assert f(fake(MIS), fake(B), fake(C), fake(D), 128, 256, 256, fake(A), 100, None) == ALIGN


def test_no_device_is_reported():
    """Valid arguments on a machine without a GPU stop at the device check."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this checks the no-device path")
    lib = binding.load()
    assert lib.jet_quant_act_1x128(fake(A), 4, 128, fake(B), fake(C), None) == DEVICE
    assert lib.jet_gemm_fp8_fwd(fake(A), fake(B), fake(C), fake(D), 128, 128, 128,
                                fake(A), None, 0, None) == DEVICE
    need = lib.jet_workspace_bytes(binding.OP["gemm_fp8_fwd"], 16, 1024, 1024)
    assert lib.jet_gemm_fp8_fwd(fake(A), fake(B), fake(C), fake(D), 16, 1024, 1024,
                                fake(A), fake(B), need, None) == DEVICE
    assert lib.jet_gemm_fp8_fwd_grouped(fake(A), fake(B), fake(C), fake(D), fake(A), 4, 256,
                                        128, 128, fake(A), None) == DEVICE
    assert lib.jet_swiglu_quant_1x128(fake(A), fake(B), 512, 4, 256, fake(C), fake(D),
                                      None) == DEVICE
    assert lib.jet_rmsnorm_quant_1x128(fake(A), fake(B), 4, 256, 1e-5, fake(C), fake(D),
                                       None) == DEVICE
    assert lib.jet_token_mismatch_per_sequence(fake(A), fake(B), None, fake(D), 4, 16, 0.0, None,
                                               fake(C), None, None) == DEVICE
    assert lib.jet_kv_calibrate(fake(A), 4, 8, 128, fake(B), None) == DEVICE
    assert lib.jet_kv_cache_write(fake(A), fake(B), fake(C), 4, 8, 128, fake(D), 16,
                                  None) == DEVICE
    for name in ("jet_gemm_fp8_dgrad_grouped", "jet_gemm_fp8_wgrad_grouped"):
        assert getattr(lib, name)(fake(A), fake(B), fake(C), fake(D), fake(A), 4, 256, 128,
                                  128, fake(A), None) == DEVICE
    assert lib.jet_device_status(None, None) == DEVICE


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    """No silent fallback: a missing library raises instead of computing elsewhere."""
    monkeypatch.setattr(binding._build, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(ImportError):
        binding.load(build_if_missing=False)
