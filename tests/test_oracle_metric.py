"""Pins for the oracle's token-mult-prob-error (CPU only).

The metric is (1/n) * sum_i exp(|logp_train_i - logp_infer_i|) ("NVIDIA强化学习加速
实操：10分钟提升2倍训练效率", section "FP8面临的关键挑战：数值分歧").  Pins: equal
inputs give exactly 1; a constant gap d gives e^d; symmetry; and the closed form
E[e^|d|] = 2 e^(sigma^2/2) Phi(sigma) for d ~ N(0, sigma^2), checked at n = 4M.
"""
import math

import numpy as np

import oracle
from fp8_block_quantized_gb300 import workloads as wl
from tests.golden_io import load_metric_band


def test_equal_inputs_give_one():
    a = np.random.default_rng(0).standard_normal(1000).astype(np.float32)
    assert oracle.token_mult_prob_error(a, a) == 1.0


def test_constant_gap():
    rng = np.random.default_rng(1)
    b = np.log(rng.uniform(1e-4, 1, 4096)).astype(np.float64)
    for d in (0.01, 0.25, 2.0):
        a = (b + d).astype(np.float32)
        bb = b.astype(np.float32)
        exact = np.mean(np.exp(np.abs(a.astype(np.float64) - bb.astype(np.float64))))
        r = oracle.token_mult_prob_error(a, bb)
        assert abs(r - exact) <= 1e-12 * exact              # summation order only
        assert abs(r - math.exp(d)) < 1e-5 * math.exp(d)   # binary32 inputs


def test_symmetry_and_sign_mix():
    rng = np.random.default_rng(2)
    b = rng.standard_normal(2048).astype(np.float32)
    d = np.where(np.arange(2048) % 2 == 0, 0.5, -0.5).astype(np.float32)
    a = b + d
    r1 = oracle.token_mult_prob_error(a, b)
    r2 = oracle.token_mult_prob_error(b, a)
    assert r1 == r2


def test_closed_form_gaussian_gap():
    sigma = 0.02
    n = 4_194_304
    a, b = wl.logprobs(n)
    r = oracle.token_mult_prob_error(a.numpy(), b.numpy())
    phi = 0.5 * (1 + math.erf(sigma / math.sqrt(2)))
    expect = 2 * math.exp(sigma ** 2 / 2) * phi            # 1.0161598...
    assert abs(expect - 1.0161598) < 5e-8
    assert abs(r - expect) < 3e-5                           # ~5 standard errors
    lo, hi = load_metric_band()
    assert r < lo < hi                                      # sigma = 0.02 sits below the band


# ---------------------------------------------- masked metric + IS weights --

def test_masked_metric_all_tokens_equals_plain_metric():
    rng = np.random.default_rng(11)
    a = rng.normal(-2, 1, 5000).astype(np.float32)
    b = (a + rng.normal(0, 0.05, 5000)).astype(np.float32)
    m, c, _ = oracle.token_mismatch_masked(a, b)
    assert c == 5000
    assert abs(m - oracle.token_mult_prob_error(a, b)) <= 1e-15 * m
    m1, c1, _ = oracle.token_mismatch_masked(a, b, np.ones(5000, np.uint8))
    assert (m1, c1) == (m, c)


def test_masked_metric_closed_form_on_masked_tokens():
    """Masked tokens differ by exactly d, the others by anything: metric = e^|d|."""
    rng = np.random.default_rng(12)
    n = 4096
    mask = (rng.random(n) < 0.37).astype(np.uint8)
    # multiples of 2^-10 in (-8, 0]: b + d is exact in binary32
    b = (np.round(rng.uniform(-8, 0, n) * 1024) / 1024).astype(np.float32)
    d = np.float32(-0.375)
    a = np.where(mask == 1, b + d, rng.normal(0, 3, n)).astype(np.float32)
    assert (a[mask == 1] - b[mask == 1] == d).all()
    m, c, w = oracle.token_mismatch_masked(a, b, mask)
    assert c == int(mask.sum())
    assert abs(m - math.exp(0.375)) <= 1e-12          # summation of equal terms only
    assert np.allclose(w[mask == 1], math.exp(-0.375), rtol=1e-15, atol=0)
    assert (w[mask == 0] == 0).all()


def test_importance_weights_direction_and_cap():
    """w = p_train / p_rollout: a token the rollout model found less likely
    than the trained model gets weight > 1 (the pages' correction raises it)."""
    b = np.log(np.array([0.5, 0.01, 0.2, 0.9], np.float32))        # rollout
    a = np.log(np.array([0.5, 0.05, 0.1, 0.9], np.float32))        # train
    _, _, w = oracle.token_mismatch_masked(a, b)
    ratio = np.exp(a.astype(np.float64) - b.astype(np.float64))
    assert np.allclose(w, ratio, rtol=1e-15)
    assert w[0] == 1.0 and w[3] == 1.0
    assert w[1] > 1.0 and w[2] < 1.0
    assert abs(w[1] - 5.0) < 1e-5 and abs(w[2] - 0.5) < 1e-6
    _, _, wc = oracle.token_mismatch_masked(a, b, cap=2.0)
    assert wc[1] == 2.0 and np.array_equal(wc[[0, 2, 3]], w[[0, 2, 3]])
    _, _, wz = oracle.token_mismatch_masked(a, b, cap=0.0)        # no cap
    assert np.array_equal(wz, w)


def test_masked_metric_subset_and_empty():
    rng = np.random.default_rng(13)
    a = rng.normal(-3, 1, 1000).astype(np.float32)
    b = (a + rng.normal(0, 0.1, 1000)).astype(np.float32)
    mask = np.zeros(1000, np.uint8)
    mask[::3] = 1
    m, c, _ = oracle.token_mismatch_masked(a, b, mask)
    assert c == 334
    direct = np.mean(np.exp(np.abs(a[::3].astype(np.float64) - b[::3].astype(np.float64))))
    assert abs(m - direct) <= 1e-14 * direct
    m0, c0, w0 = oracle.token_mismatch_masked(a, b, np.zeros(1000, np.uint8))
    assert c0 == 0 and math.isnan(m0) and (w0 == 0).all()


def test_per_sequence_metric_pins():
    """Per-sequence metrics: one sequence is the masked metric over all
    tokens; the count-weighted mean of the sequences' metrics is that metric;
    a constant gap d in a sequence gives e^|d|; an empty or fully masked-out
    sequence gives NaN with count 0."""
    rng = np.random.default_rng(9)
    lens = np.array([5, 0, 130, 1, 64, 17])
    off = np.concatenate([[0], np.cumsum(lens)])
    n = int(off[-1])
    b = np.log(rng.uniform(1e-4, 1, n)).astype(np.float32)
    a = (b + rng.normal(0, 0.05, n)).astype(np.float32)
    mask = (rng.uniform(size=n) < 0.7).astype(np.uint8)
    mask[off[4]:off[5]] = 0                       # sequence 4 fully masked out
    r, c, w = oracle.token_mismatch_per_sequence(a, b, off, mask, cap=2.0)
    whole, count, w_all = oracle.token_mismatch_masked(a, b, mask, cap=2.0)
    assert np.array_equal(w, w_all)
    ok = c > 0
    assert np.isclose((r[ok] * c[ok]).sum() / c.sum(), whole, rtol=1e-14)
    assert c.sum() == count and c[1] == 0 and c[4] == 0
    assert np.isnan(r[1]) and np.isnan(r[4])
    one, cnt1, _ = oracle.token_mismatch_per_sequence(a, b, np.array([0, n]), mask, cap=2.0)
    assert one[0] == whole and cnt1[0] == count
    d = np.float32(0.25)
    bb = np.zeros(10, np.float32) - 3.0
    aa = bb + d
    rr, cc, _ = oracle.token_mismatch_per_sequence(aa, bb, np.array([0, 4, 10]))
    dd = float(np.float64(aa[0]) - np.float64(bb[0]))
    assert np.allclose(rr, [np.exp(abs(dd))] * 2, rtol=1e-15) and cc.tolist() == [4, 6]
