"""GPU parity of token-mult-prob-error against the FP64 oracle (relative 1e-5),
and the bounded-wait failure path (a wait nothing completes times out, the
status is reported, the context stays usable)."""
import math

import numpy as np
import pytest
import torch

import oracle
from fp8_block_quantized_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jet(torch_cuda):
    import fp8_block_quantized_gb300 as j
    j.load()
    return j


def check(jet, a, b, rtol=1e-5):
    r = jet.token_mult_prob_error(a.cuda(), b.cuda())
    ref = oracle.token_mult_prob_error(a.numpy(), b.numpy())
    got = float(r.cpu()[0])
    assert abs(got - ref) <= rtol * ref, (got, ref)
    return got, ref


def test_metric_4m_tokens(jet):
    a, b = wl.logprobs(4_194_304)
    got, ref = check(jet, a, b)
    sigma = 0.02
    expect = 2 * math.exp(sigma ** 2 / 2) * 0.5 * (1 + math.erf(sigma / math.sqrt(2)))
    assert abs(got - expect) < 3e-5


@pytest.mark.parametrize("n", [1, 3, 4, 5, 1000, 2047, 2049, 8192, 100_003])
def test_metric_sizes(jet, n):
    a, b = wl.logprobs(n, seed=n)
    check(jet, a, b)


def test_metric_equal_inputs_exactly_one(jet):
    a, _ = wl.logprobs(123_457)
    assert float(jet.token_mult_prob_error(a.cuda(), a.cuda()).cpu()[0]) == 1.0


def test_metric_large_gaps(jet):
    g = torch.Generator().manual_seed(3)
    b = torch.randn(50_000, generator=g)
    a = b + torch.randn(50_000, generator=g) * 2.0
    check(jet, a, b)


def test_bounded_wait_times_out_and_context_survives(jet):
    code, word = jet.device_status()
    assert code == 0 and word == 0
    jet.selftest_bounded_wait(20_000)             # 20 ms limit on a barrier nobody completes
    code, word = jet.device_status()
    assert code == 7, (code, word)                # JET_ERR_TIMEOUT
    assert (word & 0xFF) == 7 and (word >> 8) == 99
    code, word = jet.device_status()              # reading clears it
    assert code == 0 and word == 0
    a, b = wl.logprobs(4096)
    check(jet, a, b)                              # the context is still usable
