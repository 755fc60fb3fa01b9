"""Pins for the oracle's binary64 GEMMs (CPU only).

Checked against: a pure-Python triple loop on tiny shapes, numpy float64
matmul of the dequantized matrices (PyTorch's E4M3 table), the exact identity
case W = 448*I (every weight block gets s = 1 and code 0x7E on the diagonal,
so Y = dq(X) * 448 exactly), and the transposition relations between the
forward, dgrad and wgrad definitions.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_quantized_gb300 import workloads as wl

TAB = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def dq_rows(q, s):
    """Dequantize a [R, C] tensor whose scales are [C/128, R] (1x128 groups)."""
    return TAB[q] * np.repeat(s.astype(np.float64), 128, axis=0).T


def dq_blocks(q, s):
    """Dequantize a [R, C] tensor with 128x128 block scales [R/128, C/128]."""
    return TAB[q] * np.kron(s.astype(np.float64), np.ones((128, 128)))


def dq_cols(qT, sT):
    """Dequantize a [C, R] tensor whose scales are [R/128, C] (128x1 groups)."""
    return TAB[qT] * np.repeat(sT.astype(np.float64), 128, axis=0).T


def rand_q(rng, shape):
    q = rng.integers(0, 0x7F, size=shape).astype(np.uint8)
    return q | (rng.integers(0, 2, size=shape).astype(np.uint8) << 7)


def rel_err(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


def test_fwd_triple_loop_tiny():
    rng = np.random.default_rng(0)
    M, N, K = 3, 128, 256
    qx, qw = rand_q(rng, (M, K)), rand_q(rng, (N, K))
    sx = rng.uniform(0.01, 2, (K // 128, M)).astype(np.float32)
    sw = rng.uniform(0.01, 2, (N // 128, K // 128)).astype(np.float32)
    y = oracle.gemm_fwd(qx, sx, qw, sw)
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += (TAB[qx[m, k]] * float(sx[k // 128, m])) * \
                       (TAB[qw[n, k]] * float(sw[n // 128, k // 128]))
            assert abs(y[m, n] - acc) <= 1e-12 * max(abs(acc), 1e-30)


def test_fwd_dgrad_wgrad_vs_numpy_matmul():
    rng = np.random.default_rng(1)
    M, N, K = 256, 384, 512
    qx, sx = rand_q(rng, (M, K)), rng.uniform(1e-3, 1, (K // 128, M)).astype(np.float32)
    qw, sw = rand_q(rng, (N, K)), rng.uniform(1e-3, 1, (N // 128, K // 128)).astype(np.float32)
    qdy, sdy = rand_q(rng, (M, N)), rng.uniform(1e-5, 1e-2, (N // 128, M)).astype(np.float32)
    X, W, dY = dq_rows(qx, sx), dq_blocks(qw, sw), dq_rows(qdy, sdy)
    assert rel_err(oracle.gemm_fwd(qx, sx, qw, sw), X @ W.T) < 1e-12
    assert rel_err(oracle.gemm_dgrad(qdy, sdy, qw, sw), dY @ W) < 1e-12
    qdyT, sdyT = rand_q(rng, (N, M)), rng.uniform(1e-5, 1e-2, (M // 128, N)).astype(np.float32)
    qxT, sxT = rand_q(rng, (K, M)), rng.uniform(1e-3, 1, (M // 128, K)).astype(np.float32)
    dW = oracle.gemm_wgrad(qdyT, sdyT, qxT, sxT)
    assert dW.shape == (N, K)
    assert rel_err(dW, dq_cols(qdyT, sdyT) @ dq_cols(qxT, sxT).T) < 1e-12


def test_row_sampling_matches_full():
    rng = np.random.default_rng(2)
    M, N, K = 256, 256, 256
    qx, sx = rand_q(rng, (M, K)), rng.uniform(0.1, 1, (K // 128, M)).astype(np.float32)
    qw, sw = rand_q(rng, (N, K)), rng.uniform(0.1, 1, (N // 128, K // 128)).astype(np.float32)
    full = oracle.gemm_fwd(qx, sx, qw, sw)
    rows = np.array([255, 0, 17, 128])
    assert np.array_equal(oracle.gemm_fwd(qx, sx, qw, sw, rows=rows), full[rows])


def test_identity_weight_exact():
    c = wl.single_linear(M=128, N=256, K=256)
    qx, sx = oracle.quant_act_1x128(wl.bf16_bits(c.x))
    eye = torch.eye(256) * 448.0
    qw, sw = oracle.quant_w_128x128(wl.bf16_bits(eye.to(torch.bfloat16)))
    assert (sw == 1).all()
    y = oracle.gemm_fwd(qx, sx, qw, sw)
    assert np.array_equal(y, 448.0 * dq_rows(qx, sx))
    # dgrad with the same identity: dX = dq(dY) * 448 (W symmetric)
    assert np.array_equal(oracle.gemm_dgrad(qx, sx, qw, sw), 448.0 * dq_rows(qx, sx))


def test_transposition_relations():
    """wgrad(dY^T, X^T) == (dgrad-like) dq(dY)^T @ dq(X) on the requantized operands."""
    c = wl.single_linear(M=256, N=256, K=384)
    qx, sx = oracle.quant_act_1x128(wl.bf16_bits(c.x))
    qdy, sdy = oracle.quant_act_1x128(wl.bf16_bits(c.dy))
    qxT, sxT = oracle.requant_128x1(qx, sx)
    qdyT, sdyT = oracle.requant_128x1(qdy, sdy)
    dW = oracle.gemm_wgrad(qdyT, sdyT, qxT, sxT)
    ref = dq_cols(qdyT, sdyT) @ dq_cols(qxT, sxT).T
    assert dW.shape == (256, 384)
    assert rel_err(dW, ref) < 1e-12
    # and the requantized operands stay close to the unquantized product
    Xf = c.x.double().numpy()
    dYf = c.dy.double().numpy()
    exact = dYf.T @ Xf
    assert rel_err(dW, exact) < 0.1


def test_grouped_forward_is_per_expert_forward():
    """Expert e's rows use only expert e's tokens and weights; an expert with
    no tokens contributes nothing; a single expert is the plain forward."""
    rng = np.random.default_rng(5)
    E, N, K = 4, 256, 384
    counts = np.array([3, 0, 130, 7])
    off = np.concatenate([[0], np.cumsum(counts)])
    Mt = int(off[-1])
    qx = rand_q(rng, (Mt, K))
    sx = rng.uniform(0.01, 1, (K // 128, Mt)).astype(np.float32)
    qw = rand_q(rng, (E, N, K))
    sw = rng.uniform(0.01, 1, (E, N // 128, K // 128)).astype(np.float32)
    y = oracle.gemm_fwd_grouped(qx, sx, qw, sw, off)
    assert y.shape == (Mt, N)
    for e in range(E):
        a, b = off[e], off[e + 1]
        if b > a:
            ref = dq_rows(qx[a:b], sx[:, a:b]) @ dq_blocks(qw[e], sw[e]).T
            assert rel_err(y[a:b], ref) < 1e-12
    # swapping two experts' weights changes exactly their rows
    qw2, sw2 = qw.copy(), sw.copy()
    qw2[[0, 3]], sw2[[0, 3]] = qw[[3, 0]], sw[[3, 0]]
    y2 = oracle.gemm_fwd_grouped(qx, sx, qw2, sw2, off)
    assert np.array_equal(y2[off[1]:off[3]], y[off[1]:off[3]])
    assert not np.allclose(y2[:off[1]], y[:off[1]])
    one = oracle.gemm_fwd_grouped(qx[:3], sx[:, :3].copy(), qw[:1], sw[:1], np.array([0, 3]))
    assert np.array_equal(one, oracle.gemm_fwd(qx[:3], sx[:, :3].copy(), qw[0], sw[0]))


def test_grouped_dgrad_is_per_expert_dgrad():
    rng = np.random.default_rng(6)
    E, N, K = 3, 256, 384
    off = np.array([0, 129, 129, 200])
    Mt = int(off[-1])
    qdy = rand_q(rng, (Mt, N))
    sdy = rng.uniform(0.01, 1, (N // 128, Mt)).astype(np.float32)
    qw = rand_q(rng, (E, N, K))
    sw = rng.uniform(0.01, 1, (E, N // 128, K // 128)).astype(np.float32)
    dx = oracle.gemm_dgrad_grouped(qdy, sdy, qw, sw, off)
    assert dx.shape == (Mt, K)
    for e in range(E):
        a, b = off[e], off[e + 1]
        if b > a:
            ref = dq_rows(qdy[a:b], sdy[:, a:b]) @ dq_blocks(qw[e], sw[e])
            assert rel_err(dx[a:b], ref) < 1e-12
    one = oracle.gemm_dgrad_grouped(qdy, sdy, qw[2:3], sw[2:3], np.array([0, Mt]))
    assert np.array_equal(one, oracle.gemm_dgrad(qdy, sdy, qw[2], sw[2]))


def test_grouped_wgrad_is_per_expert_wgrad_and_sums_to_wgrad():
    """Expert e's dW uses only its own token blocks; an expert without tokens
    gets zeros; the experts' dW add up to the WGrad over all tokens."""
    rng = np.random.default_rng(7)
    N, K = 128, 256
    off = np.array([0, 256, 256, 384, 768])
    E, Mt = off.size - 1, int(off[-1])
    qdyT = rand_q(rng, (N, Mt))
    sdyT = rng.uniform(0.01, 1, (Mt // 128, N)).astype(np.float32)
    qxT = rand_q(rng, (K, Mt))
    sxT = rng.uniform(0.01, 1, (Mt // 128, K)).astype(np.float32)
    dw = oracle.gemm_wgrad_grouped(qdyT, sdyT, qxT, sxT, off)
    assert dw.shape == (E, N, K)
    assert (dw[1] == 0).all()
    for e in range(E):
        a, b = off[e], off[e + 1]
        if b > a:
            ref = (dq_cols(qdyT[:, a:b], sdyT[a // 128:b // 128])
                   @ dq_cols(qxT[:, a:b], sxT[a // 128:b // 128]).T)
            assert rel_err(dw[e], ref) < 1e-12
    total = oracle.gemm_wgrad(qdyT, sdyT, qxT, sxT)
    assert rel_err(dw.sum(axis=0), total) < 1e-12
    with pytest.raises(ValueError):
        oracle.gemm_wgrad_grouped(qdyT, sdyT, qxT, sxT, np.array([0, 100, 768]))
