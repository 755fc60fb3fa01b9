"""Pins of the oracle's RMSNorm fused with the 1x128 quantizer.

The pages fuse RMSNorm into custom kernels ("Jet-RL ..." gist.science,
"Implementierung") and quantize a linear layer's input in the operator that
produces it (163.com, section 五), without arithmetic; the oracle evaluates
y = x * g / sqrt(mean(x^2) + eps) in binary32 in one fixed order, then applies
the 1x128 group rule to y.  Nothing here retypes that order.  The pins:

* y is within the first-order rounding bound of that evaluation of binary64
  RMSNorm (each partial sum adds K/32 squares, five butterfly additions,
  then a division, an addition, a square root, a reciprocal and two products);
* rows of +-2^j with eps = 0 normalise exactly to +-1, so the result equals the
  (separately pinned) 1x128 quantizer applied to sign(x) * g, bit for bit;
* with eps = 0 scaling x by a power of two changes nothing, and scaling g by
  2^j scales every group scale by 2^j and leaves the codes;
* a worked group computed by hand: K = 128, x = 3 everywhere, eps = 0;
* zero rows give scale 1 and zero codes (the sign of zero kept); rows are
  independent; a wrong eps or a dropped half of the row fails the bound."""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_quantized_gb300 import workloads as wl

U = 2.0 ** -24


def bf16(t):
    return wl.bf16_bits(t.to(torch.bfloat16))


def gain(K, seed=0):
    g = torch.Generator().manual_seed(seed)
    return (1.0 + 0.1 * torch.randn(K, generator=g)).to(torch.bfloat16)


def rms64(xb, gb, eps):
    x = xb.view(np.int16).astype(np.int32) << 16
    x = x.astype(np.uint32).view(np.float32).astype(np.float64)
    g = (gb.view(np.int16).astype(np.int32) << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    e = np.float64(np.float32(eps))
    return x * g / np.sqrt((x * x).mean(axis=1, keepdims=True) + e)


def bound(K):
    """First-order relative rounding bound of the binary32 evaluation."""
    return ((K // 32 + 5) / 2 + 6) * U


@pytest.mark.parametrize("K,eps", [(128, 1e-5), (384, 1e-6), (4096, 1e-5), (5120, 1e-6),
                                   (14336, 1e-5)])
def test_within_bound_of_binary64(K, eps):
    x = bf16(wl.activations(6, K, seed=K, config=7).float())
    g = bf16(gain(K, seed=K))
    y = oracle.rmsnorm_f32(x, g, eps).astype(np.float64)
    ref = rms64(x, g, eps)
    nz = ref != 0
    rel = np.abs(y[nz] - ref[nz]) / np.abs(ref[nz])
    assert rel.max() <= bound(K), rel.max() / U


def test_small_rows_see_eps():
    """A row far below sqrt(eps) is x * g / sqrt(eps): the eps term is used."""
    K, eps = 256, 1e-2
    x = bf16(1e-4 * torch.randn(2, K, generator=torch.Generator().manual_seed(1)))
    g = bf16(gain(K))
    y = oracle.rmsnorm_f32(x, g, eps).astype(np.float64)
    ref = rms64(x, g, eps)
    assert np.max(np.abs(y - ref) / np.abs(ref).clip(1e-300)) <= bound(K)
    ref_no_eps = rms64(x, g, 0.0)
    assert np.max(np.abs(y - ref_no_eps) / np.abs(ref_no_eps)) > 0.5   # eps matters here


def test_dropping_half_the_row_breaks_the_bound():
    """The pin is sharp enough to see a sum of squares over half the row."""
    K = 4096
    x = bf16(wl.activations(3, K, seed=5, config=7).float())
    g = bf16(gain(K))
    half = x.copy()
    half[:, K // 2:] = 0
    y_half = oracle.rmsnorm_f32(half, g, 1e-5)[:, :K // 2].astype(np.float64)
    ref = rms64(x, g, 1e-5)[:, :K // 2]
    assert np.max(np.abs(y_half - ref) / np.abs(ref).clip(1e-300)) > 100 * bound(K)


@pytest.mark.parametrize("j", [-6, 0, 3])
def test_unit_rows_reduce_to_the_plain_quantizer(j):
    """x = +-2^j, eps = 0: mean(x^2) = 4^j exactly, sqrt = 2^j, r = 2^-j,
    y = sign(x) * g exactly; the result is the 1x128 quantizer of sign(x)*g."""
    K = 1024
    rng = np.random.default_rng(j + 10)
    sign = np.where(rng.random((5, K)) < 0.5, -1.0, 1.0)
    x = bf16(torch.from_numpy(sign * 2.0 ** j))
    g = gain(K, seed=3)
    q, s = oracle.rmsnorm_quant_1x128(x, bf16(g), 0.0)
    q0, s0 = oracle.quant_act_1x128(bf16(torch.from_numpy(sign) * g.float()))
    assert np.array_equal(q, q0)
    assert np.array_equal(s.view(np.uint32), s0.view(np.uint32))


@pytest.mark.parametrize("j", [-20, -3, 5, 20])
def test_power_of_two_scaling_of_x_changes_nothing(j):
    K = 2048
    x = wl.activations(4, K, seed=2, config=7).float()
    g = bf16(gain(K, seed=2))
    q, s = oracle.rmsnorm_quant_1x128(bf16(x), g, 0.0)
    q2, s2 = oracle.rmsnorm_quant_1x128(bf16(x * 2.0 ** j), g, 0.0)
    assert np.array_equal(q, q2)
    assert np.array_equal(s.view(np.uint32), s2.view(np.uint32))


@pytest.mark.parametrize("j", [-4, 2])
def test_power_of_two_gain_scales_the_scales(j):
    K = 1024
    x = bf16(wl.activations(4, K, seed=3, config=7).float())
    g = gain(K, seed=4)
    q, s = oracle.rmsnorm_quant_1x128(x, bf16(g), 1e-5)
    q2, s2 = oracle.rmsnorm_quant_1x128(x, bf16(g * 2.0 ** j), 1e-5)
    assert np.array_equal(q, q2)
    assert np.array_equal(s2, (s * np.float32(2.0 ** j)).astype(np.float32))


def test_worked_group_by_hand():
    """K = 128, x = 3 everywhere, eps = 0: sum of squares 1152 (exact), mean
    9, sqrt 3, r = RN(1/3) = 0x3EAAAAAB, 3 * r = 1.0000000298 -> RN = 1.0, so
    y = g exactly.  With g = 1 except g[7] = 2 and g[9] = -0.5: amax 2,
    s = RN(2/448) = RN(1/224), and the codes are E4(1/s), E4(2/s), E4(-0.5/s)."""
    K = 128
    x = bf16(torch.full((1, K), 3.0))
    gv = torch.ones(K)
    gv[7], gv[9] = 2.0, -0.5
    q, s = oracle.rmsnorm_quant_1x128(x, bf16(gv), 0.0)
    s_hand = np.float32(2.0) / np.float32(448.0)
    assert s[0, 0] == s_hand
    # 2 / s = 448 -> 0x7E; 1 / s = 224 -> 0x76 (224 = 1.75 * 2^7: e = 14, m = 6);
    # -0.5 / s = -112 -> 0xEE (112 = 1.75 * 2^6: e = 13, m = 6, sign set)
    assert q[0, 7] == 0x7E and q[0, 0] == 0x76 and q[0, 9] == 0xEE
    assert (np.delete(q[0], [7, 9]) == 0x76).all()


def test_zero_rows():
    K = 256
    x = np.zeros((3, K), np.uint16)
    x[1] = 0x8000                                   # -0 everywhere
    xf = wl.activations(1, K, seed=9, config=7)
    x[2] = bf16(xf)[0]
    g = bf16(gain(K))
    for eps in (1e-5, 0.0):
        q, s = oracle.rmsnorm_quant_1x128(x, g, eps)
        assert (q[0] == 0).all() and (s[:, 0] == 1.0).all()
        assert (q[1] == 0x80).all() and (s[:, 1] == 1.0).all()
        assert (s[:, 2] != 1.0).all()


def test_rows_independent():
    K = 512
    x = bf16(wl.activations(9, K, seed=6, config=7).float())
    g = bf16(gain(K))
    q, s = oracle.rmsnorm_quant_1x128(x, g, 1e-5)
    q1, s1 = oracle.rmsnorm_quant_1x128(x[4:7], g, 1e-5)
    assert np.array_equal(q[4:7], q1) and np.array_equal(s[:, 4:7], s1)
