"""jet_token_mult_prob_error_noalloc: the metric for callers that cannot
allocate device memory (the library keeps the partial sums in its own static
device array).  Called through the C ABI with raw device pointers and
compared with jet_token_mult_prob_error (caller-supplied workspace), which
launches the same kernels on the same grid and sums in the same fixed order,
so the two must agree bit for bit; also compared with the oracle's binary64
metric within the metric's tolerance, and called once through the Python
binding.  Two calls in a row with different inputs, so that the second call
(fewer blocks) runs over the first call's leftover scratch contents.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process."""
import ctypes

import pytest
import torch

import oracle
from fp8_block_quantized_gb300 import binding
from fp8_block_quantized_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

RTOL = 1e-5
MAX_TOKENS = 2_097_152


def raw(t):
    return ctypes.c_void_p(t.data_ptr())


def reference_value(lib, a, b, stream):
    n = a.numel()
    ws = torch.empty((max(lib.jet_workspace_bytes(6, n, 0, 0), 16),), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty((1,), dtype=torch.float32, device="cuda")
    assert lib.jet_token_mult_prob_error(raw(a), raw(b), n, raw(out), raw(ws),
                                         ws.numel(), stream) == 0
    return out


def test_noalloc_matches_workspace_version_twice(torch_cuda):
    lib = binding.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [wl.logprobs(MAX_TOKENS, seed=11), wl.logprobs(300_001, seed=12)]
    outs = []
    for a_h, b_h in cases:                   # two calls in a row
        a, b = a_h.cuda(), b_h.cuda()
        out = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
        code = lib.jet_token_mult_prob_error_noalloc(raw(a), raw(b), a.numel(), raw(out), stream)
        assert code == 0, binding.STATUS.get(code, code)
        ref = reference_value(lib, a, b, stream)
        torch.cuda.synchronize()
        # same kernels, grid and summation order: identical bits
        assert out.view(torch.int32).item() == ref.view(torch.int32).item(), \
            (out.item(), ref.item())
        want = oracle.token_mult_prob_error(a_h.numpy(), b_h.numpy())
        got = float(out.item())
        assert abs(got - want) <= RTOL * want, (got, want)
        # the Python binding's wrapper reaches the same entry point
        out2 = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
        binding.jet_token_mult_prob_error_noalloc(a, b, out2)
        torch.cuda.synchronize()
        assert out2.view(torch.int32).item() == out.view(torch.int32).item()
        outs.append(got)
    assert outs[0] != outs[1]
    code, word = binding.device_status()
    assert code == 0, (code, word)


def test_noalloc_rejects_sizes_beyond_its_scratch(torch_cuda):
    lib = binding.load()
    a, b = (t.cuda() for t in wl.logprobs(64))
    out = torch.empty((1,), dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.jet_token_mult_prob_error_noalloc(raw(a), raw(b), MAX_TOKENS + 1, raw(out),
                                                 stream) == 2          # JET_ERR_SHAPE
    assert lib.jet_token_mult_prob_error_noalloc(raw(a), raw(b), 0, raw(out), stream) == 2
