"""Pins for the oracle's fused SwiGLU + 1x128 quantizer (CPU only).

The binary32 exp and silu are pinned against binary64 mathematics (ulp
bounds over dense sweeps, exact limits); the grouping and scaling are pinned
by reduction to the already pinned 1x128 activation quantizer (with up = 1
and gates where silu(g) = g exactly) and by exact symmetries."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def all_bf16(lo, hi):
    b = np.arange(0, 1 << 16, dtype=np.uint32)
    f = (b << 16).view(np.float32)
    return f[np.isfinite(f) & (f >= lo) & (f <= hi)]


def ulps(got, ref):
    """|got - ref| in units of the binary32 spacing at |ref| (ref binary64)."""
    sp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    return np.abs(got.astype(np.float64) - ref) / sp


def test_exp_within_one_ulp():
    x = np.concatenate([np.linspace(-87, 80, 400_001), all_bf16(-87, 80)]).astype(np.float32)
    e = oracle.exp_f32(x)
    assert ulps(e, np.exp(x.astype(np.float64))).max() <= 1.0
    assert oracle.exp_f32(np.float32(0.0)) == 1.0


def test_exp_subnormal_range_and_underflow():
    x = np.linspace(-103.9, -87.5, 2001).astype(np.float32)
    e = oracle.exp_f32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    # results below 2^-126 are subnormal: absolute error within one subnormal step
    assert (np.abs(e - ref) <= 2.0 ** -149).all()


def test_silu_within_three_ulps():
    g = all_bf16(-80, 80)
    ref = g.astype(np.float64) / (1.0 + np.exp(-g.astype(np.float64)))
    got = oracle.silu_f32(g)
    keep = np.abs(ref) > 1e-30
    assert ulps(got[keep], ref[keep]).max() <= 3.0
    assert (np.abs(got[~keep].astype(np.float64) - ref[~keep]) <= 1e-36).all()


def test_silu_limits_and_signed_zeros():
    g = all_bf16(17, 3.4e38)                       # e^-g below half an ulp of 1
    assert np.array_equal(oracle.silu_f32(g), g)
    neg = all_bf16(-3.4e38, -80.5)
    out = oracle.silu_f32(neg)
    assert (out == 0).all() and np.signbit(out).all()
    z = oracle.silu_f32(np.array([0.0, -0.0], np.float32))
    assert z[0] == 0 and not np.signbit(z[0]) and z[1] == 0 and np.signbit(z[1])
    # silu(1) = 1 / (1 + 1/e)
    assert ulps(oracle.silu_f32(np.float32(1.0)).reshape(1), np.array([1 / (1 + np.exp(-1.0))]))[0] <= 3


def bf16(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_reduces_to_activation_quantizer():
    """up = 1 and gates >= 17 (silu(g) = g exactly): the same codes and scales
    as the 1x128 activation quantizer of the gates."""
    rng = np.random.default_rng(3)
    M, F = 37, 384
    g = (17.0 + rng.exponential(200.0, (M, F))).astype(np.float32)
    g[5, :128] = 448.0
    gb = bf16(g)
    ub = bf16(np.ones((M, F), np.float32))
    q, s = oracle.swiglu_quant_1x128(gb, ub)
    q_ref, s_ref = oracle.quant_act_1x128(gb)
    assert np.array_equal(q, q_ref) and np.array_equal(s.view(np.uint32), s_ref.view(np.uint32))


def test_zero_up_and_sign_symmetry():
    rng = np.random.default_rng(4)
    M, F = 19, 256
    gb = bf16(rng.standard_normal((M, F)) * 3)
    ub = bf16(rng.standard_normal((M, F)))
    q, s = oracle.swiglu_quant_1x128(gb, ub)
    # negating up negates h exactly: same scales, sign bits flipped
    qn, sn = oracle.swiglu_quant_1x128(gb, ub ^ np.uint16(0x8000))
    assert np.array_equal(qn, q ^ 0x80) and np.array_equal(sn, s)
    q0, s0 = oracle.swiglu_quant_1x128(gb, np.zeros_like(ub))
    assert (s0 == 1.0).all() and np.isin(q0, [0x00, 0x80]).all()


def test_rows_and_groups_are_independent():
    rng = np.random.default_rng(5)
    M, F = 23, 512
    gb = bf16(rng.standard_normal((M, F)) * 2)
    ub = bf16(rng.standard_normal((M, F)))
    q, s = oracle.swiglu_quant_1x128(gb, ub)
    perm = rng.permutation(M)
    qp, sp = oracle.swiglu_quant_1x128(gb[perm], ub[perm])
    assert np.array_equal(qp, q[perm]) and np.array_equal(sp, s[:, perm])
    q2, s2 = oracle.swiglu_quant_1x128(gb[:, 256:384], ub[:, 256:384])
    assert np.array_equal(q2, q[:, 256:384]) and np.array_equal(s2[0], s[2])


def test_reciprocal_seed_constant_is_the_balanced_linear_seed():
    """The seed 0x7EF311C7 - bits(d) of the silu's reciprocal is the
    bit-pattern seed whose relative error over a binade equioscillates:
    about +-5.05%, equal at both ends to 1e-5, so that three Newton steps
    (error squared each time) leave 1/d to below 1e-10 in exact arithmetic.
    Any other constant nearby unbalances the two extremes."""
    d = np.linspace(1.0, 4.0, 3_000_001, dtype=np.float32)  # two binades
    def seed_err(c):
        y = (np.uint32(c) - d.view(np.uint32)).view(np.float32).astype(np.float64)
        return y * d.astype(np.float64) - 1.0
    e = seed_err(0x7EF311C7)
    assert 0.0504 < e.max() < 0.0506 and -0.0506 < e.min() < -0.0504
    assert abs(e.max() + e.min()) < 1e-5
    for c in (0x7EF00000, 0x7EF80000):
        f = seed_err(c)
        assert abs(f.max() + f.min()) > 1e-3
    assert np.abs(e).max() ** 8 < 1e-10
