"""GPU parity of the three quantizers against the CPU oracle: codes and scales
bit-exact, called through the C ABI.  Inputs are the seeded workloads (and
edge cases); the oracle quantizes the same host copy.  Large inputs are checked
on sampled row / block-row / column-block slices, which the oracle computes
independently because groups never straddle them."""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_quantized_gb300 import workloads as wl
from tests.gpu_util import assert_codes_equal, assert_scales_equal, bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jet(torch_cuda):
    import fp8_block_quantized_gb300 as j
    j.load()
    return j


def check_act(jet, x_cpu, rows=None):
    q, s = jet.quant_act_1x128(x_cpu.cuda())
    torch.cuda.synchronize()
    xb = bits(x_cpu)
    if rows is None:
        q_ref, s_ref = oracle.quant_act_1x128(xb)
        assert_codes_equal(q, q_ref)
        assert_scales_equal(s, s_ref)
    else:
        q_ref, s_ref = oracle.quant_act_1x128(xb[rows])
        assert_codes_equal(q[torch.as_tensor(rows).cuda()], q_ref)
        assert_scales_equal(s[:, torch.as_tensor(rows).cuda()], s_ref)


def test_act_single_linear(jet):
    c = wl.single_linear()
    check_act(jet, c.x)
    check_act(jet, c.dy)


@pytest.mark.parametrize("M", [1, 16, 17, 64, 65, 256, 2048])
@pytest.mark.parametrize("K", [128, 4096, 14336])
def test_act_rollout_shapes(jet, M, K):
    check_act(jet, wl.activations(M, K, seed=M + K, config=2))


def test_act_edge_values(jet):
    M, K = 70, 384
    x = torch.zeros((M, K), dtype=torch.float32)
    x[1] = 3.3895e38                                     # BF16 max
    x[2, :128] = torch.linspace(-1e-38, 1e-38, 128)      # subnormal range
    x[3] = -0.0
    x[4, :] = 448.0
    x[4, 7] = 17.0                                       # ties
    x[5] = torch.arange(K) * (2.0 ** -10)
    x[6] = -torch.arange(K).float()
    TAB = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float()
    codes = torch.randint(0, 0x7F, (K,), generator=torch.Generator().manual_seed(1))
    x[7] = TAB[codes] * torch.where(torch.arange(K) % 3 == 0, -1.0, 1.0)
    x[7, ::128] = 448.0                                  # representable, scale 1
    x[8:] = torch.randn((M - 8, K), generator=torch.Generator().manual_seed(2)) * 1e-3
    check_act(jet, x.to(torch.bfloat16))


def test_act_empty(jet):
    q, s = jet.quant_act_1x128(torch.empty((0, 256), dtype=torch.bfloat16, device="cuda"))
    assert q.shape == (0, 256) and s.shape == (2, 0)


def test_act_train8b_full_sampled_rows(jet):
    x = wl.activations(8192, 14336, seed=0, config=3, tensor_id=3)
    rows = np.sort(np.random.default_rng(0).choice(8192, 1024, replace=False))
    rows[-1] = 8191
    check_act(jet, x, rows)


def test_act_sync_heavy_activation_full_sampled_rows(jet):
    """The weight-sync sweep's 16384 x 14336 Student-t(3) activation matrix."""
    x = wl.heavy_activations(16384, 14336, seed=0)
    rows = np.sort(np.random.default_rng(3).choice(16384, 1024, replace=False))
    rows[0], rows[-1] = 0, 16383
    check_act(jet, x, rows)


def test_act_heavy_tailed_gradients(jet):
    dy = wl.grad_output(8192, 1024, seed=0, config=3, tensor_id=201)
    check_act(jet, dy)


def check_w(jet, w_cpu, block_rows=None):
    q, s = jet.quant_w_128x128(w_cpu.cuda())
    torch.cuda.synchronize()
    wb = bits(w_cpu)
    if block_rows is None:
        q_ref, s_ref = oracle.quant_w_128x128(wb)
        assert_codes_equal(q, q_ref)
        assert_scales_equal(s, s_ref)
    else:
        for nb in block_rows:
            sl = slice(nb * 128, (nb + 1) * 128)
            q_ref, s_ref = oracle.quant_w_128x128(wb[sl])
            assert_codes_equal(q[sl], q_ref)
            assert_scales_equal(s[nb:nb + 1], s_ref)


def test_w_single_linear(jet):
    check_w(jet, wl.single_linear().w)


@pytest.mark.parametrize("N,K", [(128, 128), (1024, 4096), (4096, 14336), (384, 640)])
def test_w_shapes(jet, N, K):
    check_w(jet, wl.weights(N, K, seed=N ^ K, config=5))


def test_w_gate_sampled_block_rows(jet):
    check_w(jet, wl.weights(14336, 4096, seed=0, config=5, tensor_id=104), [0, 5, 57, 111])


@pytest.mark.parametrize("layer", [0, 13, 31])
def test_w_sync_layer_every_weight_sampled(jet, layer):
    """Weight sync (the 32-layer 8B model's weights, seeded as the sync
    workload draws them): every one of the layer's 7 weights, 3 block rows
    each (the first, the last and one in between), bit-exact."""
    for i, (name, N, K) in enumerate(wl.LLAMA8B_LINEARS):
        w = wl.weights(N, K, seed=0, config=5, tensor_id=1000 + 10 * layer + i)
        nb = N // 128
        check_w(jet, w, sorted({0, (layer * 7 + i * 13) % nb, nb - 1}))


def test_w_identity_and_zero(jet):
    w = torch.zeros((256, 256))
    w[:128, :128] = torch.eye(128) * 448.0
    check_w(jet, w.to(torch.bfloat16))


def check_requant(jet, x_cpu, kblocks=None):
    q_ref, s_ref = oracle.quant_act_1x128(bits(x_cpu))
    M, K = q_ref.shape
    qT, sT = jet.requant_128x1(to_dev(q_ref), to_dev(s_ref))
    torch.cuda.synchronize()
    if kblocks is None:
        qT_ref, sT_ref = oracle.requant_128x1(q_ref, s_ref)
        assert_codes_equal(qT, qT_ref)
        assert_scales_equal(sT, sT_ref)
    else:
        for kb in kblocks:
            sl = slice(kb * 128, (kb + 1) * 128)
            qT_ref, sT_ref = oracle.requant_128x1(np.ascontiguousarray(q_ref[:, sl]),
                                                  np.ascontiguousarray(s_ref[kb:kb + 1]))
            assert_codes_equal(qT[sl], qT_ref)
            assert_scales_equal(sT[:, sl], sT_ref)


def test_requant_single_linear(jet):
    c = wl.single_linear()
    check_requant(jet, c.x)
    check_requant(jet, c.dy)


@pytest.mark.parametrize("M,K", [(128, 128), (384, 256), (1024, 1024)])
def test_requant_shapes(jet, M, K):
    check_requant(jet, wl.activations(M, K, seed=M * 7 + K, config=3, zero_group=True))


def test_requant_gradients_train8b_sampled(jet):
    dy = wl.grad_output(8192, 4096, seed=0, config=3, tensor_id=200)
    check_requant(jet, dy, kblocks=[0, 13, 31])


def test_requant_empty(jet):
    qT, sT = jet.requant_128x1(torch.empty((0, 128), dtype=torch.uint8, device="cuda"),
                               torch.empty((1, 0), dtype=torch.float32, device="cuda"))
    assert qT.shape == (128, 0) and sT.shape == (0, 128)


def check_dual(jet, x_cpu, kblocks=None):
    """The fused quantizer against the oracle's 1x128 quantization followed by
    its 128x1 re-quantization of the FP8 values."""
    q, s, qT, sT = jet.quant_dual_1x128_128x1(x_cpu.cuda())
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_act_1x128(bits(x_cpu))
    assert_codes_equal(q, q_ref)
    assert_scales_equal(s, s_ref)
    if kblocks is None:
        qT_ref, sT_ref = oracle.requant_128x1(q_ref, s_ref)
        assert_codes_equal(qT, qT_ref)
        assert_scales_equal(sT, sT_ref)
    else:
        for kb in kblocks:
            sl = slice(kb * 128, (kb + 1) * 128)
            qT_ref, sT_ref = oracle.requant_128x1(np.ascontiguousarray(q_ref[:, sl]),
                                                  np.ascontiguousarray(s_ref[kb:kb + 1]))
            assert_codes_equal(qT[sl], qT_ref)
            assert_scales_equal(sT[:, sl], sT_ref)


def test_dual_single_linear(jet):
    c = wl.single_linear()
    check_dual(jet, c.dy)
    check_dual(jet, c.x)      # outlier channels and an all-zero 1x128 group


@pytest.mark.parametrize("M,K", [(128, 128), (384, 256), (1024, 1024), (256, 14336)])
def test_dual_shapes(jet, M, K):
    check_dual(jet, wl.grad_output(M, K, seed=M * 3 + K, config=3))


def test_dual_edge_values(jet):
    M, K = 256, 384
    x = torch.randn((M, K), generator=torch.Generator().manual_seed(3)) * 1e-3
    x[:, 5] = 0.0                                   # an all-zero 128x1 group per token block
    x[7, :] = -0.0                                   # signed zeros
    x[9, 128:256] = 3.3895e38                        # BF16 max in one group
    x[200:, 300] = 1e-38                             # subnormal column
    check_dual(jet, x.to(torch.bfloat16))


def test_dual_train8b_gradients_sampled(jet):
    check_dual(jet, wl.grad_output(8192, 4096, seed=0, config=3, tensor_id=200), kblocks=[0, 17, 31])


def test_dual_empty(jet):
    q, s, qT, sT = jet.quant_dual_1x128_128x1(torch.empty((0, 256), dtype=torch.bfloat16, device="cuda"))
    assert q.shape == (0, 256) and qT.shape == (256, 0) and sT.shape == (0, 256)


def _ieee_quotients(x, s):
    with np.errstate(all="ignore"):
        return (x.astype(np.float32) / s.astype(np.float32)).astype(np.float32)


def test_division_routine_matches_ieee(jet):
    """The quantizers' group division equals IEEE binary32 x / s where codes
    can depend on it (and always in sign, with tiny quotients below 2^-10)."""
    rng = np.random.default_rng(42)
    n = 4_000_000
    # x across the whole binary32 range, signed, with zeros and subnormals
    x = (rng.standard_normal(n) * np.exp2(rng.uniform(-150, 100, n))).astype(np.float32)
    x[::97] = 0.0
    x[1::97] = -0.0
    # s = fl32(amax / 448) with amax >= |x| in the same group sense
    amax = (np.abs(x).astype(np.float64) * np.exp2(rng.uniform(0, 20, n))).astype(np.float32)
    amax = np.maximum(amax, np.float32(1e-44))
    s = (amax / np.float32(448)).astype(np.float32)
    s[s == 0] = np.float32(1.0)
    # boundary cases: quotients within a few ulps of every E4M3 rounding midpoint
    tab = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()[:0x7F]
    mids = ((tab[:-1] + tab[1:]) / 2).astype(np.float32)
    sb = (np.exp2(rng.uniform(-80, 100, mids.size * 64)) / 448).astype(np.float32)
    mb = np.repeat(mids, 64)
    xb = (mb.astype(np.float64) * sb.astype(np.float64)).astype(np.float32)
    steps = rng.integers(-3, 4, xb.size).astype(np.int32)
    xb = (xb.view(np.int32) + steps).view(np.float32)
    x = np.concatenate([x, xb, -xb])
    s = np.concatenate([s, sb, sb])
    q = jet.selftest_quotient(torch.from_numpy(x).cuda(), torch.from_numpy(s).cuda())
    got = q.cpu().numpy()
    want = _ieee_quotients(x, s)
    exact_region = (s < np.float32(2.0 ** -90)) | (np.abs(want) >= np.float32(2.0 ** -11))
    bad = np.flatnonzero(exact_region & (got.view(np.uint32) != want.view(np.uint32)))
    assert bad.size == 0, (bad.size, x[bad[:3]], s[bad[:3]], got[bad[:3]], want[bad[:3]])
    tiny = ~exact_region
    assert (np.signbit(got[tiny]) == np.signbit(want[tiny])).all()
    assert (np.abs(got[tiny]) < np.float32(2.0 ** -10)).all()
    assert exact_region.sum() > 0.3 * x.size


def test_act_near_division_fast_path_threshold(jet):
    """Groups whose scale sits on either side of the fast-path threshold."""
    M, K = 64, 256
    rng = np.random.default_rng(5)
    x = rng.standard_normal((M, K)).astype(np.float32)
    amax_target = np.float32(448.0 * 2.0 ** -90) * np.exp2(rng.uniform(-3, 3, (M, 1))).astype(np.float32)
    x = x / np.abs(x).max(axis=1, keepdims=True) * amax_target
    check_act(jet, torch.from_numpy(x).to(torch.bfloat16))


# ------------------------------------------------ SwiGLU + 1x128, fused --

def check_swiglu(jet, g_cpu, u_cpu, fused=False, rows=None):
    """The fused SwiGLU quantizer against the oracle's binary32 SwiGLU and
    1x128 group rule; `fused` passes gate and up as the two halves of one
    [M, 2F] tensor (the layout of a gate_up product)."""
    M, F = g_cpu.shape
    if fused:
        gu = torch.cat([g_cpu, u_cpu], dim=1).cuda()
        q, s = jet.swiglu_quant_1x128(gu[:, :F], gu[:, F:])
    else:
        q, s = jet.swiglu_quant_1x128(g_cpu.cuda(), u_cpu.cuda())
    torch.cuda.synchronize()
    gb, ub = bits(g_cpu), bits(u_cpu)
    if rows is None:
        q_ref, s_ref = oracle.swiglu_quant_1x128(gb, ub)
        assert_codes_equal(q, q_ref, "swiglu codes")
        assert_scales_equal(s, s_ref, "swiglu scales")
    else:
        q_ref, s_ref = oracle.swiglu_quant_1x128(gb[rows], ub[rows])
        r = torch.as_tensor(rows).cuda()
        assert_codes_equal(q[r], q_ref, "swiglu codes")
        assert_scales_equal(s[:, r], s_ref, "swiglu scales")


@pytest.mark.parametrize("M,F", [(1, 128), (37, 384), (256, 768), (300, 1536), (130, 14336)])
@pytest.mark.parametrize("fused", [False, True])
def test_swiglu_shapes(jet, M, F, fused):
    g = wl.activations(M, F, seed=M + F, config=6, tensor_id=30)
    u = wl.activations(M, F, seed=M + F, config=6, tensor_id=31)
    check_swiglu(jet, g * 3, u, fused=fused)


def test_swiglu_edge_values(jet):
    M, F = 64, 384
    gen = torch.Generator().manual_seed(11)
    g = torch.randn((M, F), generator=gen) * 4
    u = torch.randn((M, F), generator=gen)
    g[0] = -100.0                                  # silu -> signed zero
    g[1, :128] = torch.linspace(-90, -70, 128)     # across the -80 cut
    g[2] = 0.0
    g[3] = -0.0
    u[4] = 0.0                                     # all-zero groups: scale 1
    g[5] = 1e4                                     # silu(g) = g
    u[5] = torch.linspace(-3, 3, F)
    g[6, :] = torch.linspace(-104.5, 104.5, F)     # both clamps of the exponent
    g[7] = 1e-38                                   # subnormal products
    u[7] = 1e-3
    g[8, ::2] = 30.0
    u[8, ::2] = 14.9                               # exact products, ties in E4M3
    check_swiglu(jet, g.to(torch.bfloat16), u.to(torch.bfloat16))
    check_swiglu(jet, g.to(torch.bfloat16), u.to(torch.bfloat16), fused=True)


def test_swiglu_every_bf16_gate(jet):
    """Every finite BF16 gate value (65,280 of them) through the binary32
    sequence, with up = 1 and up = -1.5; the gates sorted in 128-groups so
    that most groups span a narrow range and small values set their scale."""
    b = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    v = b.view(torch.bfloat16).float()
    v = v[torch.isfinite(v)]
    v = v[torch.argsort(v)]
    n = (v.numel() // 128) * 128
    g = v[:n].view(-1, 128).to(torch.bfloat16)
    for up in (1.0, -0.75):
        check_swiglu(jet, g, torch.full_like(g, up))


def test_swiglu_moe_sized_sampled(jet):
    g = wl.activations(32768, 768, seed=0, config=6, tensor_id=32)
    u = wl.activations(32768, 768, seed=0, config=6, tensor_id=33)
    rows = np.sort(np.random.default_rng(1).choice(32768, 2048, replace=False))
    rows[-1] = 32767
    check_swiglu(jet, g, u, fused=True, rows=rows)


def test_swiglu_empty(jet):
    e = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    q, s = jet.swiglu_quant_1x128(e, e)
    assert q.shape == (0, 256) and s.shape == (2, 0)


# ----------------------------------------------- RMSNorm + 1x128, fused --

def check_rmsnorm(jet, x_cpu, g_cpu, eps, rows=None):
    """The fused RMSNorm quantizer against the oracle's binary32 RMSNorm (its
    fixed order of operations) and 1x128 group rule: codes and scales bit for
    bit."""
    q, s = jet.rmsnorm_quant_1x128(x_cpu.cuda(), g_cpu.cuda(), eps)
    torch.cuda.synchronize()
    xb, gb = bits(x_cpu), bits(g_cpu)
    if rows is None:
        q_ref, s_ref = oracle.rmsnorm_quant_1x128(xb, gb, eps)
        assert_codes_equal(q, q_ref, "rmsnorm codes")
        assert_scales_equal(s, s_ref, "rmsnorm scales")
    else:
        q_ref, s_ref = oracle.rmsnorm_quant_1x128(xb[rows], gb, eps)
        r = torch.as_tensor(rows).cuda()
        assert_codes_equal(q[r], q_ref, "rmsnorm codes")
        assert_scales_equal(s[:, r], s_ref, "rmsnorm scales")


@pytest.mark.parametrize("M,K", [(1, 128), (37, 384), (300, 1024), (129, 4096), (64, 5120),
                                 (16, 8192), (9, 14336), (3, 25600)])
@pytest.mark.parametrize("eps", [1e-5, 1e-6])
def test_rmsnorm_shapes(jet, M, K, eps):
    x = wl.activations(M, K, seed=M + K, config=3, tensor_id=40)
    check_rmsnorm(jet, x, wl.norm_gain(K, seed=K), eps)


def test_rmsnorm_edge_values(jet):
    M, K = 40, 512
    gen = torch.Generator().manual_seed(12)
    x = torch.randn((M, K), generator=gen)
    x[0] = 0.0                                     # zero row: r = 1/sqrt(eps)
    x[1] = -0.0
    x[2] = 1e-30                                   # tiny rows: eps dominates
    x[3, :] = 3.0                                  # exact normalisation
    x[4] = 1e17                                    # large (the sum stays finite)
    x[5, :128] = 0.0                               # an all-zero group in a live row
    x[6] = torch.linspace(-7, 7, K)
    x[7, ::2] = 448.0
    g = (1.0 + 0.1 * torch.randn(K, generator=gen))
    g[::17] = -g[::17]                             # negative gains
    g[5] = 0.0
    for eps in (1e-5, 0.0):
        check_rmsnorm(jet, x.to(torch.bfloat16), g.to(torch.bfloat16), eps)


def test_rmsnorm_train32b_sampled(jet):
    """The 32B layer's attention input at full size (16384 x 5120)."""
    x = wl.activations(16384, 5120, seed=0, config=4, tensor_id=0)
    rows = np.sort(np.random.default_rng(4).choice(16384, 1024, replace=False))
    rows[0], rows[-1] = 0, 16383
    check_rmsnorm(jet, x, wl.norm_gain(5120, seed=0, config=4), 1e-6, rows)


def test_rmsnorm_empty(jet):
    e = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    g = torch.ones((256,), dtype=torch.bfloat16, device="cuda")
    q, s = jet.rmsnorm_quant_1x128(e, g)
    assert q.shape == (0, 256) and s.shape == (2, 0)
