"""GPU parity of the GEMM paths that only the 32B-shaped training layer
(hidden 5120, M = 16384 tokens) takes, against the oracle's FP64 product of the
same dequantized operands (|Y - ref| <= 2^-7 |ref| + 1e-3 rms(ref row)):

* the down projection's forward (Y [16384, 5120], contraction 25600 = 200
  slices) and the gate projection's DGrad (contraction 25600): both operands
  are larger than the L2 budget of the tile order, so the tiles run in groups
  of column tiles (20 column tiles in groups of 7, 7 and 6);
* the same products at 4224 rows (17 row tiles, the last one's second CTA
  entirely past the last row);
* the o projection's DGrad and the down projection's WGrad (dW rows: 20 row
  tiles in two groups of 10).

The operands are the oracle's own quantization of the seeded layer tensors
(the tensor ids of the 32B training layer), copied to the device; the
outputs are checked on whole rows: one row in each 128-row half of every
256-row pair tile (so every tile of the output, whatever the tile order, is
checked in both CTAs of its pair), the first and last rows, and random ones.
("Jet-RL ..." gist.science summary, "Quantisierungsschema": forward, DGrad
and WGrad in FP8.)"""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_quantized_gb300 import workloads as wl
from tests.gpu_util import assert_gemm_close, bits, pair_tile_rows, to_dev

pytestmark = pytest.mark.gpu

M32 = 16384
CFG = wl.CONFIG_ID["train32b"]
# tensor ids of the 32B layer (workloads.training_layer): distinct inputs
# 0 attn_in, 1 attn_out, 2 mlp_in, 3 mlp_act; weights 100 + i, dY 200 + i
# for the linears in order q, k, v, o, gate, up, down
_cache = {}


@pytest.fixture(scope="module")
def jet(torch_cuda):
    import fp8_block_quantized_gb300 as j
    j.load()
    return j


def cached(key, make):
    if key not in _cache:
        _cache[key] = make()
    return _cache[key]


def w_quant(name):
    """Oracle 128x128 quantization of one 32B weight (numpy codes, scales)."""
    idx = [n for n, _, _ in wl.DENSE32B_LINEARS].index(name)
    _, N, K = wl.DENSE32B_LINEARS[idx]
    return cached(("w", name), lambda: oracle.quant_w_128x128(
        bits(wl.weights(N, K, seed=0, config=CFG, tensor_id=100 + idx))))


def x_quant(tensor_id, K, M=M32):
    return cached(("x", tensor_id, M), lambda: oracle.quant_act_1x128(
        bits(wl.activations(M, K, seed=0, config=CFG, tensor_id=tensor_id))))


def dy_quant(name, M=M32):
    idx = [n for n, _, _ in wl.DENSE32B_LINEARS].index(name)
    _, N, _ = wl.DENSE32B_LINEARS[idx]
    return cached(("dy", name, M), lambda: oracle.quant_act_1x128(
        bits(wl.grad_output(M, N, seed=0, config=CFG, tensor_id=200 + idx))))


def checked_rows(M, extra, k=16, seed=0):
    """k random rows plus the given rows."""
    r = np.random.default_rng(seed).choice(M, k, replace=False)
    return np.unique(np.concatenate([r, np.asarray([x for x in extra if x < M])]))


def check(out, ref, rows, what):
    assert_gemm_close(out[torch.as_tensor(rows).cuda()], ref, what)


def test_train32b_down_fwd_raster_groups(jet):
    """Y = X W_down^T: 16384 x 5120 over K = 25600 (200 slices)."""
    qx, sx = x_quant(3, 25600)
    qw, sw = w_quant("down")
    y = jet.gemm_fp8_fwd(to_dev(qx), to_dev(sx), to_dev(qw), to_dev(sw))
    torch.cuda.synchronize()
    rows = checked_rows(M32, pair_tile_rows(M32))
    check(y, oracle.gemm_fwd(qx, sx, qw, sw, rows=rows), rows, "down fwd 32B")


def test_train32b_gate_dgrad_raster_groups(jet):
    """dX = dY_gate W_gate: 16384 x 5120 over N = 25600."""
    qdy, sdy = dy_quant("gate")
    qw, sw = w_quant("gate")
    dx = jet.gemm_fp8_dgrad(to_dev(qdy), to_dev(sdy), to_dev(qw), to_dev(sw))
    torch.cuda.synchronize()
    rows = checked_rows(M32, pair_tile_rows(M32, 1), seed=1)
    check(dx, oracle.gemm_dgrad(qdy, sdy, qw, sw, rows=rows), rows, "gate dgrad 32B")


@pytest.mark.parametrize("M", [4224])
def test_short_last_raster_group(jet, M):
    """17 pair tiles of rows, the last one's second CTA entirely past the
    last row, for the forward and the DGrad of the widest contraction
    (column groups of 7, 7 and 6)."""
    qx, sx = x_quant(3, 25600, M=M)
    qw, sw = w_quant("down")
    y = jet.gemm_fp8_fwd(to_dev(qx), to_dev(sx), to_dev(qw), to_dev(sw))
    qdy, sdy = dy_quant("gate", M=M)
    qg, sg = w_quant("gate")
    dx = jet.gemm_fp8_dgrad(to_dev(qdy), to_dev(sdy), to_dev(qg), to_dev(sg))
    torch.cuda.synchronize()
    rows = checked_rows(M, pair_tile_rows(M, 2) + list(range(4096, 4224, 9)), k=8, seed=2)
    check(y, oracle.gemm_fwd(qx, sx, qw, sw, rows=rows), rows, "fwd, short group")
    check(dx, oracle.gemm_dgrad(qdy, sdy, qg, sg, rows=rows), rows, "dgrad, short group")


def test_train32b_o_dgrad(jet):
    """dX = dY_o W_o: 16384 x 8192 over N = 5120."""
    qdy, sdy = dy_quant("o")
    qw, sw = w_quant("o")
    dx = jet.gemm_fp8_dgrad(to_dev(qdy), to_dev(sdy), to_dev(qw), to_dev(sw))
    torch.cuda.synchronize()
    rows = checked_rows(M32, [0, 255, M32 - 1], seed=3)
    check(dx, oracle.gemm_dgrad(qdy, sdy, qw, sw, rows=rows), rows, "o dgrad 32B")


def test_train32b_down_wgrad(jet):
    """dW = dY_down^T X: 5120 x 25600 over the 16384 tokens (128 token
    groups), operands re-quantized 128x1 from their 1x128 form."""
    qx, sx = x_quant(3, 25600)
    qdy, sdy = dy_quant("down")
    qxT, sxT = cached(("xT", 3), lambda: oracle.requant_128x1(qx, sx))
    qdyT, sdyT = oracle.requant_128x1(qdy, sdy)
    dw = jet.gemm_fp8_wgrad(to_dev(qdyT), to_dev(sdyT), to_dev(qxT), to_dev(sxT))
    torch.cuda.synchronize()
    rows = checked_rows(5120, pair_tile_rows(5120, 4), seed=4)
    check(dw, oracle.gemm_wgrad(qdyT, sdyT, qxT, sxT, rows=rows), rows, "down wgrad 32B")
