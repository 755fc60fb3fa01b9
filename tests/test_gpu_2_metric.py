"""GPU parity of token-mult-prob-error against the FP64 oracle (relative 1e-5),
and the bounded-wait failure path (a wait nothing completes times out, the
status is reported, the context stays usable)."""
import math

import numpy as np
import pytest
import torch

import oracle
from fp8_block_quantized_gb300 import workloads as wl
from tests.gpu_util import assert_gemm_close

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


def test_gemm_timeout_path_and_context_survives(jet):
    """The GEMM's own failure path: with its pipeline waits limited to a few
    hundred SM cycles (shorter than the first operand load from memory), a
    role of the single-CTA kernel gives up, records a GEMM wait site, the
    others stop, loads and MMAs drain and TMEM is freed; afterwards the same
    product at the normal limit matches the oracle, and so does a larger
    product that fills every SM (TMEM was released everywhere)."""
    x = wl.activations(128, 1024, seed=31, config=1)
    w = wl.weights(512, 1024, seed=31, config=1)
    qx, sx = oracle.quant_act_1x128(wl.bf16_bits(x))
    qw, sw = oracle.quant_w_128x128(wl.bf16_bits(w))
    dq = [torch.from_numpy(a).cuda() for a in (qx, sx, qw, sw)]
    code, word = jet.device_status()
    assert code == 0 and word == 0
    for limit in (64, 300):
        # fresh operands in DRAM each time (not in L2): evict with a write
        torch.empty(256 << 20, dtype=torch.uint8, device="cuda").fill_(1)
        jet.selftest_gemm_timeout(*dq, limit)
        code, word = jet.device_status()
        assert code == 7, (limit, code, word)                 # JET_ERR_TIMEOUT
        assert (word >> 8) in (1, 2, 3, 4), hex(word)         # a GEMM wait site
        assert jet.device_status() == (0, 0)                  # reading clears it
    y = jet.selftest_gemm_timeout(*dq, 4_000_000_000)          # the library's own limit
    assert jet.device_status() == (0, 0)
    assert_gemm_close(y, oracle.gemm_fwd(qx, sx, qw, sw), "fwd after time-outs")
    xb = wl.activations(4096, 1024, seed=32, config=1)
    wb = wl.weights(2048, 1024, seed=32, config=1)
    qxb, sxb = oracle.quant_act_1x128(wl.bf16_bits(xb))
    qwb, swb = oracle.quant_w_128x128(wl.bf16_bits(wb))
    yb = jet.gemm_fp8_fwd(*(torch.from_numpy(a).cuda() for a in (qxb, sxb, qwb, swb)))
    assert jet.device_status() == (0, 0)
    rows = np.arange(0, 4096, 97)
    assert_gemm_close(yb[torch.as_tensor(rows).cuda()], oracle.gemm_fwd(qxb, sxb, qwb, swb, rows=rows),
                      "fwd on every SM after time-outs")



# ---------------------------------------------- masked metric + IS weights --

def check_masked(jet, a, b, mask=None, cap=0.0, rtol=1e-5, wtol=2e-6):
    """Metric within 1e-5 relative of the oracle; weights within a few FP32
    ulps (expf of the FP32 difference against binary64); count exact."""
    dev_mask = None if mask is None else torch.from_numpy(mask).cuda()
    out, count, w = jet.token_mismatch_masked(a.cuda(), b.cuda(), dev_mask, cap)
    ref, ref_count, ref_w = oracle.token_mismatch_masked(a.numpy(), b.numpy(), mask, cap)
    got = float(out.cpu()[0])
    assert int(count.cpu()[0]) == ref_count
    if ref_count == 0:
        assert math.isnan(got)
    else:
        assert abs(got - ref) <= rtol * ref, (got, ref)
    gw = w.cpu().numpy().astype(np.float64)
    on = ref_w != 0
    assert (gw[~on] == 0).all()
    assert np.allclose(gw[on], ref_w[on], rtol=wtol, atol=0), np.max(np.abs(gw[on] / ref_w[on] - 1))
    if cap > 0:
        assert (gw <= np.float32(cap)).all()
    return got, ref


@pytest.mark.parametrize("n", [1, 3, 4, 5, 2047, 2049, 100_003])
def test_masked_sizes(jet, n):
    a, b = wl.logprobs(n, seed=n)
    mask = (np.random.default_rng(n).random(n) < 0.8).astype(np.uint8)
    mask[0] = 1
    check_masked(jet, a, b, mask)


def test_masked_4m_tokens_with_cap(jet):
    a, b = wl.logprobs(4_194_304, seed=7)
    rng = np.random.default_rng(7)
    mask = np.ones(4_194_304, np.uint8)
    mask[rng.random(4_194_304) < 0.25] = 0          # prompt / padding tokens
    check_masked(jet, a, b, mask, cap=1.01)


def test_masked_without_mask_equals_plain_metric(jet):
    a, b = wl.logprobs(100_000, seed=3)
    got, _ = check_masked(jet, a, b, None)
    plain = float(jet.token_mult_prob_error(a.cuda(), b.cuda()).cpu()[0])
    assert abs(got - plain) <= 1e-6 * plain


def test_masked_no_token_counts(jet):
    a, b = wl.logprobs(1000, seed=4)
    check_masked(jet, a, b, np.zeros(1000, np.uint8))


def test_masked_optional_outputs(jet):
    """w and count may be NULL; the metric is unchanged."""
    a, b = wl.logprobs(5000, seed=5)
    mask = torch.from_numpy((np.arange(5000) % 2).astype(np.uint8)).cuda()
    out = torch.empty((1,), dtype=torch.float32, device="cuda")
    ws = torch.empty((max(jet.workspace_bytes("token_mismatch_masked", 5000), 16),),
                     dtype=torch.uint8, device="cuda")
    jet.jet_token_mismatch_masked(a.cuda(), b.cuda(), mask, 0.0, None, out, None, ws)
    ref, _, _ = oracle.token_mismatch_masked(a.numpy(), b.numpy(), mask.cpu().numpy())
    assert abs(float(out.cpu()[0]) - ref) <= 1e-5 * ref


# ---------------------------------------------------------- per sequence --

def check_per_sequence(jet, a, b, off, mask=None, cap=0.0):
    o = torch.from_numpy(np.asarray(off, np.int64)).cuda()
    m = None if mask is None else torch.from_numpy(mask).cuda()
    r, c, w = jet.token_mismatch_per_sequence(a.cuda(), b.cuda(), o, m, cap)
    r, c, w = r.cpu().numpy(), c.cpu().numpy(), w.cpu().numpy()
    rr, cc, ww = oracle.token_mismatch_per_sequence(a.numpy(), b.numpy(), off, mask, cap)
    assert np.array_equal(c, cc), "per-sequence counts"
    empty = cc == 0
    assert np.isnan(r[empty]).all()
    assert (np.abs(r[~empty] - rr[~empty]) <= 1e-5 * rr[~empty]).all(), "per-sequence metrics"
    assert np.allclose(w.astype(np.float64), ww, rtol=2e-6, atol=0), "importance weights"
    return r, c, w


def test_per_sequence_ragged_and_empty(jet):
    lens = np.array([5, 0, 130, 1, 64, 17, 0, 2049, 3])
    off = np.concatenate([[0], np.cumsum(lens)])
    n = int(off[-1])
    a, b = wl.logprobs(n, seed=11)
    mask = (np.random.default_rng(11).random(n) < 0.7).astype(np.uint8)
    mask[off[5]:off[6]] = 0                          # a fully masked-out sequence
    check_per_sequence(jet, a, b, off, mask, cap=1.02)
    check_per_sequence(jet, a, b, off, None)


def test_per_sequence_4m_tokens(jet):
    """2048 sequences of log-normal lengths (about 2048 tokens each), prompt
    tokens masked out, the weights capped."""
    rng = np.random.default_rng(12)
    lens = np.maximum(1, rng.lognormal(7.3, 0.8, 2048)).astype(np.int64)
    lens = (lens * (4_194_304 / lens.sum())).astype(np.int64)
    lens[-1] += 4_194_304 - lens.sum()
    off = np.concatenate([[0], np.cumsum(lens)])
    a, b = wl.logprobs(4_194_304, seed=12)
    mask = np.ones(4_194_304, np.uint8)
    for s in range(2048):                            # the first quarter of each sequence: prompt
        mask[off[s]:off[s] + lens[s] // 4] = 0
    check_per_sequence(jet, a, b, off, mask, cap=1.05)


def test_per_sequence_chunk_edges(jet):
    """Sequences ending and starting exactly on, and one token either side of,
    the 4096-token chunk edges, empty ones there, and one spanning chunks."""
    lens = np.array([4096, 0, 4095, 1, 1, 4094, 0, 3, 20000, 4096])
    off = np.concatenate([[0], np.cumsum(lens)])
    a, b = wl.logprobs(int(off[-1]), seed=14)
    check_per_sequence(jet, a, b, off)


def test_per_sequence_one_sequence_and_determinism(jet):
    a, b = wl.logprobs(100_003, seed=13)
    off = torch.tensor([0, 100_003], device="cuda")
    r1, c1, w1 = jet.token_mismatch_per_sequence(a.cuda(), b.cuda(), off)
    r2, _, w2 = jet.token_mismatch_per_sequence(a.cuda(), b.cuda(), off)
    assert torch.equal(r1, r2) and torch.equal(w1, w2)
    plain = float(jet.token_mult_prob_error(a.cuda(), b.cuda()).cpu()[0])
    assert abs(float(r1.cpu()[0]) - plain) <= 1e-6 * plain and int(c1.cpu()[0]) == 100_003
