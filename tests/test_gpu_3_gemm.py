"""GPU parity of the forward, DGrad and WGrad FP8 GEMMs against the oracle's
FP64 product of the same dequantized operands:

    |Y - ref| <= 2^-7 |ref| + 1e-3 * rms(ref row)   elementwise

The operands are the oracle's own quantization of the seeded workloads, copied
to the device, so each GEMM is checked on exactly the codes and scales the
oracle used.  Full-size shapes are checked on sampled output rows (the oracle
computes those rows one by one); small shapes on every element."""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_quantized_gb300 import workloads as wl
from tests.gpu_util import assert_gemm_close, bits, host, pair_tile_rows, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jet(torch_cuda):
    import fp8_block_quantized_gb300 as j
    j.load()
    return j


def quant_pair(x, w):
    qx, sx = oracle.quant_act_1x128(bits(x))
    qw, sw = oracle.quant_w_128x128(bits(w))
    return qx, sx, qw, sw


def sample_rows(n, k, seed=0):
    if n <= k:
        return None
    r = np.sort(np.random.default_rng(seed).choice(n, k, replace=False))
    r[0], r[-1] = 0, n - 1
    return np.unique(r)


def run_fwd(jet, x, w, nrows=None, rows=None):
    qx, sx, qw, sw = quant_pair(x, w)
    y = jet.gemm_fp8_fwd(to_dev(qx), to_dev(sx), to_dev(qw), to_dev(sw))
    torch.cuda.synchronize()
    if rows is None:
        rows = sample_rows(qx.shape[0], nrows) if nrows else None
    else:
        rows = np.unique(np.asarray(rows, np.int64))
    ref = oracle.gemm_fwd(qx, sx, qw, sw, rows=rows)
    assert_gemm_close(y if rows is None else y[torch.as_tensor(rows).cuda()], ref, "fwd")
    return y


def run_dgrad(jet, dy, w, nrows=None, rows=None):
    qdy, sdy = oracle.quant_act_1x128(bits(dy))
    qw, sw = oracle.quant_w_128x128(bits(w))
    dx = jet.gemm_fp8_dgrad(to_dev(qdy), to_dev(sdy), to_dev(qw), to_dev(sw))
    torch.cuda.synchronize()
    if rows is None:
        rows = sample_rows(qdy.shape[0], nrows) if nrows else None
    else:
        rows = np.unique(np.asarray(rows, np.int64))
    ref = oracle.gemm_dgrad(qdy, sdy, qw, sw, rows=rows)
    assert_gemm_close(dx if rows is None else dx[torch.as_tensor(rows).cuda()], ref, "dgrad")
    return dx


def run_wgrad(jet, dy, x, nrows=None):
    qx, sx = oracle.quant_act_1x128(bits(x))
    qdy, sdy = oracle.quant_act_1x128(bits(dy))
    qxT, sxT = oracle.requant_128x1(qx, sx)
    qdyT, sdyT = oracle.requant_128x1(qdy, sdy)
    dw = jet.gemm_fp8_wgrad(to_dev(qdyT), to_dev(sdyT), to_dev(qxT), to_dev(sxT))
    torch.cuda.synchronize()
    rows = sample_rows(qdyT.shape[0], nrows) if nrows else None
    ref = oracle.gemm_wgrad(qdyT, sdyT, qxT, sxT, rows=rows)
    assert_gemm_close(dw if rows is None else dw[torch.as_tensor(rows).cuda()], ref, "wgrad")
    return dw


# ----------------------------------------------------------- small, exact --

def test_fwd_single_tile(jet):
    run_fwd(jet, wl.activations(128, 128, seed=1, config=1), wl.weights(256, 128, seed=1, config=1))


def test_fwd_single_linear(jet):
    c = wl.single_linear()
    run_fwd(jet, c.x, c.w)


def test_dgrad_single_linear(jet):
    c = wl.single_linear()
    run_dgrad(jet, c.dy, c.w)


def test_wgrad_single_linear(jet):
    c = wl.single_linear()
    run_wgrad(jet, c.dy, c.x)


@pytest.mark.parametrize("M", [1, 16, 64, 100, 129, 256, 300, 385])
@pytest.mark.parametrize("N", [1024, 384, 128])
def test_fwd_ragged_rows_and_widths(jet, M, N):
    run_fwd(jet, wl.activations(M, 512, seed=M, config=2), wl.weights(N, 512, seed=N, config=2))


@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("N,K", [(128, 128), (256, 384), (1024, 640), (384, 1152), (4096, 14336)])
def test_fwd_decode_rows(jet, M, N, K):
    # at most 4 tokens: the weight-streaming kernel (K tails of 128 / 384 codes included)
    run_fwd(jet, wl.activations(M, K, seed=M * 7 + K, config=2), wl.weights(N, K, seed=N + K, config=2),
            nrows=None)


def test_fwd_decode_deterministic(jet):
    x, w = wl.activations(3, 4096, seed=21, config=2), wl.weights(4096, 4096, seed=21, config=2)
    qx, sx, qw, sw = (to_dev(a) for a in quant_pair(x, w))
    y1 = jet.gemm_fp8_fwd(qx, sx, qw, sw)
    y2 = jet.gemm_fp8_fwd(qx, sx, qw, sw)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(200, 256, 384), (128, 128, 256), (256, 512, 128),
                                   (384, 512, 512), (300, 256, 512)])
def test_dgrad_shapes(jet, M, N, K):
    run_dgrad(jet, wl.grad_output(M, N, seed=M + N, config=3),
              wl.weights(N, K, seed=K, config=3))


@pytest.mark.parametrize("M,N,K", [(128, 256, 384), (384, 128, 256), (256, 512, 512),
                                   (256, 384, 512)])
def test_wgrad_shapes(jet, M, N, K):
    run_wgrad(jet, wl.grad_output(M, N, seed=M + N, config=3),
              wl.activations(M, K, seed=K, config=3))


@pytest.mark.parametrize("M,N,K", [(16, 512, 1024), (1, 4096, 1024), (100, 2048, 384),
                                   (128, 4096, 1024), (256, 4096, 1024), (300, 8192, 512),
                                   (16, 4096, 4096), (16, 4096, 14336)])
def test_dgrad_small_rows_split_contraction(jet, M, N, K):
    # at most 512 rows: the contraction (N) is split into ranges of 128-slices;
    # 16 x 4096 x 4096 runs 8-slice ranges on the six-stage 128-wide kernel,
    # 16 x 4096 x 14336 (112 tiles of 128) two ranges of 256-wide tiles
    assert jet.workspace_bytes("gemm_fp8_dgrad", M, N, K) > 0
    run_dgrad(jet, wl.grad_output(M, N, seed=M + N, config=3), wl.weights(N, K, seed=K, config=3),
              nrows=None if M * K <= 16 * 4096 else 8)


@pytest.mark.parametrize("kind,M,N,K", [
    ("fwd", 50, 384, 8192),     # 128-wide ranges on six stages, ragged rows, 3 column tiles
    ("fwd", 200, 4096, 8192),   # six stages over two row tiles, the second ragged
    ("fwd", 129, 640, 8192),    # four stages, one row past the first tile
    ("dgrad", 50, 8192, 384),   # DGrad (C = K = 384) on six stages
])
def test_split_contraction_plans(jet, kind, M, N, K):
    """Decode-sized products on every kind of split kernel, ragged in rows
    and in column tiles, against the oracle on sampled rows."""
    assert jet.workspace_bytes("gemm_fp8_" + kind, M, N, K) > 0
    if kind == "fwd":
        run_fwd(jet, wl.activations(M, K, seed=M + K, config=2),
                wl.weights(N, K, seed=N + K, config=2), nrows=24)
    else:
        run_dgrad(jet, wl.grad_output(M, N, seed=M + N, config=3),
                  wl.weights(N, K, seed=K + 1, config=3), nrows=24)


def test_split_contraction_deterministic_and_workspace_agnostic(jet):
    """Same bits on repeated calls, whatever the workspace held before."""
    M, N, K = 16, 1024, 4096
    need = jet.workspace_bytes("gemm_fp8_fwd", M, N, K)
    assert need == 8 * M * N * 4  # 4 tiles: 8 contraction ranges
    x, w = wl.activations(M, K, seed=11, config=2), wl.weights(N, K, seed=11, config=2)
    qx, sx, qw, sw = (to_dev(a) for a in quant_pair(x, w))
    outs = []
    for fill in (0.0, float("nan"), 1e30):
        ws = torch.full((need // 4,), fill, dtype=torch.float32, device="cuda")
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        jet.jet_gemm_fp8_fwd(qx, sx, qw, sw, y, ws=ws)
        outs.append(y)
    torch.cuda.synchronize()
    for y in outs[1:]:
        assert torch.equal(outs[0].view(torch.int16), y.view(torch.int16))
    ref = oracle.gemm_fwd(*quant_pair(x, w))
    assert_gemm_close(outs[0], ref, "fwd split")


def test_zero_rows_are_exact_zero(jet):
    x = wl.activations(256, 384, seed=5, config=1).float()
    x[3] = 0.0
    x[200] = 0.0
    y = run_fwd(jet, x.to(torch.bfloat16), wl.weights(256, 384, seed=5, config=1))
    assert (host(y[3].float()) == 0).all() and (host(y[200].float()) == 0).all()


def test_empty_contraction_writes_zeros(jet):
    e8 = torch.empty((64, 0), dtype=torch.uint8, device="cuda")
    s = torch.empty((0, 64), dtype=torch.float32, device="cuda")
    w8 = torch.empty((256, 0), dtype=torch.uint8, device="cuda")
    sw = torch.empty((2, 0), dtype=torch.float32, device="cuda")
    y = torch.full((64, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    jet.jet_gemm_fp8_fwd(e8, s, w8, sw, y)
    assert (y == 0).all()


def test_deterministic(jet):
    x, w = wl.activations(512, 1024, seed=9, config=2), wl.weights(1024, 1024, seed=9, config=2)
    qx, sx, qw, sw = (to_dev(a) for a in quant_pair(x, w))
    y1 = jet.gemm_fp8_fwd(qx, sx, qw, sw)
    y2 = jet.gemm_fp8_fwd(qx, sx, qw, sw)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


# ----------------------------------------------- persistent, full shapes --

def test_fwd_persistent_many_tiles(jet):
    # 32 x 8 = 256 tiles > SM count: CTAs loop over several tiles
    run_fwd(jet, wl.activations(4096, 1024, seed=2, config=2), wl.weights(2048, 1024, seed=2, config=2),
            nrows=48)


@pytest.mark.parametrize("name,N,K", [("kv", 1024, 4096), ("down", 4096, 14336),
                                      ("q", 4096, 4096), ("gate", 14336, 4096)])
@pytest.mark.parametrize("M", [1, 64, 256, 385, 2048])
def test_fwd_rollout_shapes(jet, name, N, K, M):
    # every split plan appears: 128-wide ranges on six stages (q and down
    # at 64 rows, down at 256) and on four (kv; q at 256), 256-wide ranges
    # (gate at 64 rows; q and down at 385), no split on the CTA-pair kernel
    # (gate at 256 and 385 rows; everything at 2048)
    run_fwd(jet, wl.activations(M, K, seed=M, config=2), wl.weights(N, K, seed=N, config=2),
            nrows=24)


@pytest.mark.parametrize("idx", range(len(wl.LLAMA8B_LINEARS)),
                         ids=[n for n, _, _ in wl.LLAMA8B_LINEARS])
@pytest.mark.parametrize("M", [16, 2048])
def test_fwd_rollout_every_linear(jet, idx, M):
    """Each of the 7 rollout linears of the 8B layer (its own weight tensor)
    at a decode-batch and a prefill token count: split contraction at 16
    tokens, CTA pairs at 2048."""
    name, N, K = wl.LLAMA8B_LINEARS[idx]
    key = wl.SHARED_INPUT[name]
    xid = list(dict.fromkeys(wl.SHARED_INPUT[n] for n, _, _ in wl.LLAMA8B_LINEARS)).index(key)
    run_fwd(jet, wl.activations(M, K, seed=0, config=2, tensor_id=xid),
            wl.weights(N, K, seed=0, config=2, tensor_id=100 + idx), nrows=24)


def test_train8b_q_proj_fwd_dgrad_wgrad(jet):
    layer = wl.training_layer("train8b")
    q = layer[0]
    assert (q.name, q.M, q.N, q.K) == ("q", 8192, 4096, 4096)
    run_fwd(jet, q.x, q.w, nrows=24)
    run_dgrad(jet, q.dy, q.w, nrows=24)
    run_wgrad(jet, q.dy, q.x, nrows=16)


def run_wgrad_rows(jet, dy, x, rows):
    qx, sx = oracle.quant_act_1x128(bits(x))
    qdy, sdy = oracle.quant_act_1x128(bits(dy))
    qxT, sxT = oracle.requant_128x1(qx, sx)
    qdyT, sdyT = oracle.requant_128x1(qdy, sdy)
    dw = jet.gemm_fp8_wgrad(to_dev(qdyT), to_dev(sdyT), to_dev(qxT), to_dev(sxT))
    torch.cuda.synchronize()
    rows = np.unique(np.asarray(rows, np.int64))
    ref = oracle.gemm_wgrad(qdyT, sdyT, qxT, sxT, rows=rows)
    assert_gemm_close(dw[torch.as_tensor(rows).cuda()], ref, "wgrad")


def test_train8b_gate_proj_wgrad_every_pair_tile(jet):
    """dW_gate = dY^T X (14336 x 4096 over 8192 tokens): one row in each
    128-row half of every one of the 56 pair tiles of dW rows."""
    layer = wl.training_layer("train8b")
    g = layer[4]
    assert (g.name, g.M, g.N, g.K) == ("gate", 8192, 14336, 4096)
    run_wgrad_rows(jet, g.dy, g.x, pair_tile_rows(g.N, 6))


@pytest.mark.parametrize("name,N,K", [("o", 5120, 8192), ("q", 8192, 5120)])
def test_train32b_wgrad_groups_every_pair_tile(jet, name, N, K):
    """32B-layer WGrad over 16384 tokens whose operands both exceed the tile
    order's L2 budget: dW rows in groups (o: 20 row tiles in groups of 10)
    or columns in groups (q: 20 column tiles in groups of 10); one row in
    each half of every pair tile."""
    M = 16384
    idx = [n for n, _, _ in wl.DENSE32B_LINEARS].index(name)
    run_wgrad_rows(jet, wl.grad_output(M, N, seed=0, config=4, tensor_id=200 + idx),
                   wl.activations(M, K, seed=0, config=4, tensor_id=7 + idx),
                   pair_tile_rows(N, 7))


def test_train32b_kv_proj_wgrad(jet):
    M, N, K = 16384, 1024, 5120
    run_wgrad(jet, wl.grad_output(M, N, seed=0, config=4, tensor_id=201),
              wl.activations(M, K, seed=0, config=4), nrows=8)


def test_train8b_down_proj_fwd_dgrad_wgrad(jet):
    """The widest contraction of the 8B layer (K = 14336) in all three
    products.  Neither forward operand fits the tile order's L2 budget, so
    its 16 column tiles run in two groups of 8: every pair tile is checked."""
    layer = wl.training_layer("train8b")
    d = layer[6]
    assert (d.name, d.M, d.N, d.K) == ("down", 8192, 4096, 14336)
    run_fwd(jet, d.x, d.w, rows=pair_tile_rows(d.M))
    run_dgrad(jet, d.dy, d.w, nrows=16)
    run_wgrad(jet, d.dy, d.x, nrows=8)


def test_train8b_gate_proj_dgrad_column_groups(jet):
    """dX = dY_gate W_gate (8192 x 4096 over N = 14336): 16 column tiles in
    two groups of 8, every pair tile checked."""
    M, N, K = 8192, 14336, 4096
    run_dgrad(jet, wl.grad_output(M, N, seed=0, config=2, tensor_id=204),
              wl.weights(N, K, seed=0, config=2, tensor_id=104), rows=pair_tile_rows(M))


def test_fwd_short_last_row_group(jet):
    """Y = X W^T for 3712 x 3584 over K = 14336: neither operand fits the L2
    budget and the 15 row tiles (the last one's second CTA past the last
    row) run in groups of 8 and 7; every pair tile checked."""
    M, N, K = 3712, 3584, 14336
    run_fwd(jet, wl.activations(M, K, seed=1, config=2, tensor_id=3),
            wl.weights(N, K, seed=1, config=2, tensor_id=106), rows=pair_tile_rows(M, 5))


def test_train32b_gate_proj_fwd(jet):
    """The widest output of the 32B layer (N = 25600) at M = 16384."""
    M, N, K = 16384, 25600, 5120
    run_fwd(jet, wl.activations(M, K, seed=0, config=4, tensor_id=2),
            wl.weights(N, K, seed=0, config=4, tensor_id=104), nrows=8)


# ------------------------------------------ grouped forward (expert linears) --

def quant_experts(x, w):
    """Oracle quantization of the tokens and of every expert's weights."""
    qx, sx = oracle.quant_act_1x128(bits(x))
    E = w.shape[0]
    pairs = [oracle.quant_w_128x128(bits(w[e])) for e in range(E)]
    return qx, sx, np.stack([p[0] for p in pairs]), np.stack([p[1] for p in pairs])


def run_grouped(jet, x, w, off, rows_per_expert=None, experts=None):
    qx, sx, qw, sw = quant_experts(x, w)
    off = np.asarray(off, np.int64)
    y = jet.gemm_fp8_fwd_grouped(to_dev(qx), to_dev(sx), to_dev(qw), to_dev(sw),
                                 torch.from_numpy(off).cuda())
    torch.cuda.synchronize()
    if rows_per_expert is None:
        assert_gemm_close(y, oracle.gemm_fwd_grouped(qx, sx, qw, sw, off), "grouped fwd")
        return y
    # sampled rows of sampled experts: each expert's rows are the plain forward
    # product of its own tokens, which the oracle computes row by row
    for e in experts:
        a, b = int(off[e]), int(off[e + 1])
        if b == a:
            continue
        r = sample_rows(b - a, rows_per_expert, seed=e)
        r = np.arange(b - a) if r is None else r
        ref = oracle.gemm_fwd(np.ascontiguousarray(qx[a:b]), np.ascontiguousarray(sx[:, a:b]),
                              qw[e], sw[e], rows=r)
        assert_gemm_close(y[torch.as_tensor(a + r).cuda()], ref, f"grouped fwd, expert {e}")
    return y


@pytest.mark.parametrize("N", [256, 384])      # 256-wide and 128-wide column tiles
def test_grouped_ragged_and_empty_experts(jet, N):
    off = [0, 5, 5, 133, 300, 300, 301, 556, 700]   # empty, 1-row and ragged experts
    E, K = len(off) - 1, 384
    x = wl.activations(off[-1], K, seed=N, config=6)
    w = wl.weights(E * N, K, seed=N, config=6).view(E, N, K)
    run_grouped(jet, x, w, off)


def test_grouped_single_expert_is_the_forward_product(jet):
    x, w = wl.activations(300, 512, seed=3, config=6), wl.weights(256, 512, seed=3, config=6)
    y = run_grouped(jet, x, w.view(1, 256, 512), [0, 300])
    qx, sx, qw, sw = quant_pair(x, w)
    assert_gemm_close(y, oracle.gemm_fwd(qx, sx, qw, sw), "grouped, one expert")


def test_grouped_empty_leading_and_trailing_experts(jet):
    off = [0, 0, 0, 129, 129, 257, 257, 257]
    E, N, K = len(off) - 1, 256, 256
    run_grouped(jet, wl.activations(257, K, seed=4, config=6),
                wl.weights(E * N, K, seed=4, config=6).view(E, N, K), off)


def test_grouped_max_experts_one_token_each(jet):
    # 384 experts (the limit), most with one token, some with none
    rng = np.random.default_rng(8)
    counts = rng.integers(0, 3, 384)
    off = np.concatenate([[0], np.cumsum(counts)])
    E, N, K = 384, 128, 128
    run_grouped(jet, wl.activations(int(off[-1]), K, seed=8, config=6),
                wl.weights(E * N, K, seed=8, config=6).view(E, N, K), off)


def test_grouped_deterministic_and_rows_independent(jet):
    off = np.array([0, 200, 200, 650, 1000], np.int64)
    E, N, K = 4, 512, 1024
    x = wl.activations(1000, K, seed=10, config=6)
    w = wl.weights(E * N, K, seed=10, config=6).view(E, N, K)
    qx, sx, qw, sw = (to_dev(a) for a in quant_experts(x, w))
    o = torch.from_numpy(off).cuda()
    y1 = jet.gemm_fp8_fwd_grouped(qx, sx, qw, sw, o)
    y2 = jet.gemm_fp8_fwd_grouped(qx, sx, qw, sw, o)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    # expert 2 alone (its own launch) gives the same bits: tiles never mix experts
    a, b = 200, 650
    y3 = jet.gemm_fp8_fwd_grouped(qx[a:b].contiguous(), sx[:, a:b].contiguous(), qw[2:3].contiguous(),
                                  sw[2:3].contiguous(), torch.tensor([0, b - a], device="cuda"))
    assert torch.equal(y1[a:b].view(torch.int16), y3.view(torch.int16))


def test_grouped_empty_contraction_and_no_tokens(jet):
    off = torch.tensor([0, 3, 64], dtype=torch.int64, device="cuda")
    y = torch.full((64, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    jet.jet_gemm_fp8_fwd_grouped(torch.empty((64, 0), dtype=torch.uint8, device="cuda"),
                                 torch.empty((0, 64), dtype=torch.float32, device="cuda"),
                                 torch.empty((2, 256, 0), dtype=torch.uint8, device="cuda"),
                                 torch.empty((2, 2, 0), dtype=torch.float32, device="cuda"), off, y)
    assert (y == 0).all()
    y0 = jet.gemm_fp8_fwd_grouped(torch.empty((0, 128), dtype=torch.uint8, device="cuda"),
                                  torch.empty((1, 0), dtype=torch.float32, device="cuda"),
                                  torch.zeros((2, 256, 128), dtype=torch.uint8, device="cuda"),
                                  torch.ones((2, 2, 1), dtype=torch.float32, device="cuda"),
                                  torch.zeros((3,), dtype=torch.int64, device="cuda"))
    assert y0.shape == (0, 256)


@pytest.mark.parametrize("lin", [0, 1])
def test_grouped_moe_layer_sampled(jet, lin):
    """The Qwen3-30B-A3B-shaped MoE layer at full size (4096 tokens, top-8 of
    128 experts): sampled rows of sampled experts, incl. the smallest and the
    largest expert."""
    off, lins = wl.moe_layer()
    name, x, w = lins[lin]
    counts = (off[1:] - off[:-1]).numpy()
    experts = sorted({int(counts.argmin()), int(counts.argmax()), 0, 63, 127})
    run_grouped(jet, x, w, off.numpy(), rows_per_expert=6, experts=experts)


# -------------------------------------- grouped DGrad / WGrad (expert backward) --

def run_grouped_dgrad(jet, dy, w, off, rows_per_expert=None, experts=None):
    qdy, sdy = oracle.quant_act_1x128(bits(dy))
    E = w.shape[0]
    pairs = [oracle.quant_w_128x128(bits(w[e])) for e in range(E)]
    qw, sw = np.stack([p[0] for p in pairs]), np.stack([p[1] for p in pairs])
    off = np.asarray(off, np.int64)
    dx = jet.gemm_fp8_dgrad_grouped(to_dev(qdy), to_dev(sdy), to_dev(qw), to_dev(sw),
                                    torch.from_numpy(off).cuda())
    torch.cuda.synchronize()
    if rows_per_expert is None:
        assert_gemm_close(dx, oracle.gemm_dgrad_grouped(qdy, sdy, qw, sw, off), "grouped dgrad")
        return
    for e in experts:
        a, b = int(off[e]), int(off[e + 1])
        if b == a:
            continue
        r = sample_rows(b - a, rows_per_expert, seed=e)
        r = np.arange(b - a) if r is None else r
        ref = oracle.gemm_dgrad(np.ascontiguousarray(qdy[a:b]), np.ascontiguousarray(sdy[:, a:b]),
                                qw[e], sw[e], rows=r)
        assert_gemm_close(dx[torch.as_tensor(a + r).cuda()], ref, f"grouped dgrad, expert {e}")


@pytest.mark.parametrize("K", [256, 384])
def test_grouped_dgrad_ragged_and_empty_experts(jet, K):
    off = [0, 5, 5, 133, 300, 300, 301, 556, 700]
    E, N = len(off) - 1, 256
    dy = wl.grad_output(off[-1], N, seed=K, config=6)
    w = wl.weights(E * N, K, seed=K, config=6).view(E, N, K)
    run_grouped_dgrad(jet, dy, w, off)


def transposed_forms(x_bf16):
    """The oracle's 128x1 form (codes [K][M], scales [M/128][K]) of x."""
    q, s = oracle.quant_act_1x128(bits(x_bf16))
    return oracle.requant_128x1(q, s)


def run_grouped_wgrad(jet, dy, x, off, rows=None, experts=None):
    qdyT, sdyT = transposed_forms(dy)
    qxT, sxT = transposed_forms(x)
    off = np.asarray(off, np.int64)
    dw = jet.gemm_fp8_wgrad_grouped(to_dev(qdyT), to_dev(sdyT), to_dev(qxT), to_dev(sxT),
                                    torch.from_numpy(off).cuda())
    torch.cuda.synchronize()
    E = off.size - 1
    assert dw.shape == (E, qdyT.shape[0], qxT.shape[0])
    if rows is None:
        ref = oracle.gemm_wgrad_grouped(qdyT, sdyT, qxT, sxT, off)
        for e in range(E):
            if off[e + 1] == off[e]:
                assert (dw[e] == 0).all(), f"expert {e} without tokens"
            else:
                assert_gemm_close(dw[e], ref[e], f"grouped wgrad, expert {e}")
        return dw
    for e in experts:
        a, b = int(off[e]), int(off[e + 1])
        r = sample_rows(qdyT.shape[0], rows, seed=e)
        ref = oracle.gemm_wgrad(np.ascontiguousarray(qdyT[:, a:b]),
                                np.ascontiguousarray(sdyT[a // 128:b // 128]),
                                np.ascontiguousarray(qxT[:, a:b]),
                                np.ascontiguousarray(sxT[a // 128:b // 128]), rows=r)
        assert_gemm_close(dw[e][torch.as_tensor(r).cuda()], ref, f"grouped wgrad, expert {e}")
    return dw


@pytest.mark.parametrize("N,K", [(256, 256), (384, 256), (128, 384), (512, 512)])
def test_grouped_wgrad_padded_experts(jet, N, K):
    # experts padded to whole 128-token groups, two of them empty
    off = [0, 256, 256, 384, 896, 896, 1024]
    dy = wl.grad_output(off[-1], N, seed=N + K, config=6)
    x = wl.activations(off[-1], K, seed=N + K, config=6)
    run_grouped_wgrad(jet, dy, x, off)


def test_grouped_wgrad_sums_to_dense_wgrad(jet):
    """One expert over all tokens is the plain WGrad, bit for bit."""
    M, N, K = 512, 256, 256
    dy, x = wl.grad_output(M, N, seed=3, config=6), wl.activations(M, K, seed=3, config=6)
    qdyT, sdyT = (to_dev(a) for a in transposed_forms(dy))
    qxT, sxT = (to_dev(a) for a in transposed_forms(x))
    g = jet.gemm_fp8_wgrad_grouped(qdyT, sdyT, qxT, sxT, torch.tensor([0, M], device="cuda"))
    d = jet.gemm_fp8_wgrad(qdyT, sdyT, qxT, sxT)
    assert torch.equal(g[0].view(torch.int16), d.view(torch.int16))


def test_grouped_backward_empty_cases(jet):
    # no tokens at all: WGrad writes zeros for every expert
    z8 = torch.empty((256, 0), dtype=torch.uint8, device="cuda")
    zs = torch.empty((0, 256), dtype=torch.float32, device="cuda")
    dw = torch.full((2, 256, 256), 3.0, dtype=torch.bfloat16, device="cuda")
    jet.jet_gemm_fp8_wgrad_grouped(z8, zs, z8, zs, torch.zeros(3, dtype=torch.int64, device="cuda"), dw)
    assert (dw == 0).all()


def test_grouped_backward_moe_layer_sampled(jet):
    """gate_up backward of the Qwen3-30B-A3B-shaped layer at full size: DGrad
    on the routed rows, WGrad on the rows padded to whole token groups."""
    off, lins = wl.moe_layer()
    _, x, w = lins[0]
    E, N, K = w.shape
    off = off.numpy()
    counts = off[1:] - off[:-1]
    experts = sorted({int(counts.argmin()), int(counts.argmax()), 0, 77})
    dy = wl.grad_output(int(off[-1]), N, seed=0, config=6, tensor_id=210)
    run_grouped_dgrad(jet, dy, w, off, rows_per_expert=4, experts=experts)
    o = torch.from_numpy(off)
    pad = wl.moe_pad_offsets(o)
    run_grouped_wgrad(jet, wl.moe_scatter_padded(dy, o, pad), wl.moe_scatter_padded(x, o, pad),
                      pad.numpy(), rows=4, experts=experts)
