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
