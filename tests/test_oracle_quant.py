"""Pins for the oracle's three quantizers (CPU only).

Independent checks: an exact-rational nearest-code search over PyTorch's E4M3
table with binary32 quotients from numpy (brute force on small inputs), the
hand-derived groups of tests/golden/e4m3_worked_groups.txt, and invariants
that hold at any size (amax element -> +-448, all-zero group -> s = 1,
E4M3-representable inputs round-trip, power-of-two rescaling, permutation
equivariance, locality of each group as printed in the pages' table).
"""
import bisect
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from fp8_block_quantized_gb300 import workloads as wl
from tests.golden_io import load_granularity, load_worked_groups

TAB = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
POS = [Fraction(float(TAB[c])) for c in range(0x7F)]       # codes 0x00..0x7E, increasing


def brute_code(t) -> int:
    """Nearest non-negative code by exact rationals (bisection), even on ties."""
    t = np.float32(t)
    sign = 0x80 if np.signbit(t) else 0
    a = Fraction(abs(float(t)))
    if a >= 448:
        return 0x7E | sign
    i = bisect.bisect_left(POS, a)
    if i == 0:
        return sign
    lo, hi = i - 1, i
    dlo, dhi = a - POS[lo], POS[hi] - a
    c = lo if dlo < dhi else hi if dhi < dlo else (lo if lo % 2 == 0 else hi)
    return c | sign


def np_scale(amax):
    amax = np.float32(amax)
    return np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(448.0))


def brute_group(vals):
    vals = np.asarray(vals, np.float32)
    s = np_scale(np.max(np.abs(vals)))
    return s, np.array([brute_code(np.float32(v / s)) for v in vals], np.uint8)


def to_bits(x):
    return wl.bf16_bits(torch.as_tensor(x).to(torch.bfloat16))


def bf16_vals(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()


# ---------------------------------------------------------------- 1x128 ----

def test_quant_act_brute_force_small():
    x = wl.activations(4, 384, seed=3, config=1, n_outlier=2, zero_group=True)
    bits = wl.bf16_bits(x)
    q, s = oracle.quant_act_1x128(bits)
    xv = bf16_vals(bits)
    for m in range(4):
        for kb in range(3):
            sb, cb = brute_group(xv[m, kb * 128:(kb + 1) * 128])
            assert s[kb, m].view(np.uint32) == sb.view(np.uint32)
            assert np.array_equal(q[m, kb * 128:(kb + 1) * 128], cb)


def test_worked_groups_scales_and_codes():
    groups = load_worked_groups()
    for name, g in groups.items():
        x = np.zeros(128, np.float32)
        for i, (v, _) in enumerate(g["entries"]):
            x[i] = v
        bits = to_bits(x)[None, :]
        assert np.array_equal(bf16_vals(bits)[0], x), "fixture values must be BF16-exact"
        q, s = oracle.quant_act_1x128(bits)
        assert int(s[0, 0].view(np.uint32)) == g["scale_bits"], name
        want = np.zeros(128, np.uint8)
        for i, (_, c) in enumerate(g["entries"]):
            want[i] = c
        assert np.array_equal(q[0], want), name


def test_amax_maps_to_448_and_scale_bits():
    c = wl.single_linear()
    bits = wl.bf16_bits(c.x)
    q, s = oracle.quant_act_1x128(bits)
    xv = bf16_vals(bits)
    M, K = xv.shape
    g = xv.reshape(M, K // 128, 128)
    amax = np.abs(g).max(axis=2)                     # [M, Kb]
    zero = amax == 0
    assert zero.sum() == 1, "the single-linear input has exactly one all-zero group"
    exp_s = np.where(zero, np.float32(1), (amax / np.float32(448)).astype(np.float32))
    assert np.array_equal(s.T.view(np.uint32), exp_s.astype(np.float32).view(np.uint32))
    qg = q.reshape(M, K // 128, 128)
    arg = np.abs(g).argmax(axis=2)
    top = np.take_along_axis(qg, arg[..., None], axis=2)[..., 0]
    assert ((top[~zero] & 0x7F) == 0x7E).all()
    assert (qg[zero] == 0).all()


def test_representable_inputs_round_trip_and_pow2_rescale():
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 0x7F, size=(8, 256)).astype(np.uint8)
    codes |= rng.integers(0, 2, size=codes.shape).astype(np.uint8) << 7
    codes[:, 7] = 0x7E                     # every group holds +448 -> s = 1
    codes[:, 128 + 9] = 0xFE               # ... or -448
    vals = TAB[codes].astype(np.float32)
    q, s = oracle.quant_act_1x128(to_bits(vals))
    assert (s == 1.0).all()
    assert np.array_equal(q, codes)
    for j in (-20, -3, 5):                 # exact power-of-two rescaling
        qj, sj = oracle.quant_act_1x128(to_bits(vals * np.float32(2.0 ** j)))
        assert (sj == np.float32(2.0 ** j)).all()
        assert np.array_equal(qj, codes)


def test_permutation_equivariance():
    x = wl.activations(2, 256, seed=11, config=1)
    bits = wl.bf16_bits(x)
    q, s = oracle.quant_act_1x128(bits)
    perm = np.random.default_rng(0).permutation(128)
    pb = bits.copy()
    pb[:, :128] = bits[:, :128][:, perm]
    qp, sp = oracle.quant_act_1x128(pb)
    assert np.array_equal(sp, s)
    assert np.array_equal(qp[:, :128], q[:, :128][:, perm])


def test_scale_layout_is_kblock_major():
    M, K = 5, 384
    x = np.zeros((M, K), np.float32)
    for m in range(M):
        for kb in range(K // 128):
            x[m, kb * 128 + (m + kb) % 128] = 2.0 ** (m - kb)   # distinct amax per group
    q, s = oracle.quant_act_1x128(to_bits(x))
    assert s.shape == (K // 128, M)
    for m in range(M):
        for kb in range(K // 128):
            assert s[kb, m] == np.float32(2.0 ** (m - kb)) / np.float32(448)


def test_group_shapes_follow_the_pages_table():
    """Perturbing one element changes exactly the scale of its own group."""
    gran = load_granularity()
    assert gran["input_activations"] == (1, 128) and gran["output_gradients"] == (1, 128)
    assert gran["weights"] == (128, 128) and gran["wgrad_token_groups"] == (128, 1)
    rng = np.random.default_rng(9)
    x = rng.standard_normal((256, 512)).astype(np.float32)
    bits = to_bits(x)
    _, s0 = oracle.quant_act_1x128(bits)
    _, w0 = oracle.quant_w_128x128(bits)
    xb = bits.copy()
    r, c = 131, 300
    xb[r, c] = to_bits(np.array([1000.0], np.float32))[0]
    _, s1 = oracle.quant_act_1x128(xb)
    _, w1 = oracle.quant_w_128x128(xb)
    ga, gw = gran["input_activations"], gran["weights"]
    changed_a = np.argwhere(s1 != s0)
    assert changed_a.tolist() == [[c // ga[1], r // ga[0]]]
    changed_w = np.argwhere(w1 != w0)
    assert changed_w.tolist() == [[r // gw[0], c // gw[1]]]


# -------------------------------------------------------------- 128x128 ----

def test_quant_w_brute_force_small():
    w = wl.weights(256, 256, seed=2, config=1)
    bits = wl.bf16_bits(w)
    q, s = oracle.quant_w_128x128(bits)
    wv = bf16_vals(bits)
    for nb in range(2):
        for kb in range(2):
            blk = wv[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            sb, cb = brute_group(blk.reshape(-1))
            assert s[nb, kb].view(np.uint32) == sb.view(np.uint32)
            assert np.array_equal(q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128],
                                  cb.reshape(128, 128))


def test_quant_w_identity_and_zero_block():
    w = np.zeros((256, 384), np.float32)
    w[:128, :128] = np.eye(128) * 448.0
    w[128:, 256:] = np.eye(128)[:, :128] * 0.5
    q, s = oracle.quant_w_128x128(to_bits(w))
    assert s[0, 0] == 1.0 and s[0, 1] == 1.0 and s[1, 0] == 1.0      # zero blocks -> 1
    assert s[1, 2] == np.float32(0.5) / np.float32(448)
    assert np.array_equal(q[:128, :128], (np.eye(128) * 0x7E).astype(np.uint8))
    assert (q[:128, 128:] == 0).all() and (q[128:, :256] == 0).all()
    assert np.array_equal(q[128:, 256:], (np.eye(128) * 0x7E).astype(np.uint8))


# --------------------------------------------------------------- 128x1 -----

def test_requant_brute_force_small():
    x = wl.activations(256, 256, seed=4, config=1, n_outlier=3, zero_group=True)
    q, s = oracle.quant_act_1x128(wl.bf16_bits(x))
    qT, sT = oracle.requant_128x1(q, s)
    assert qT.shape == (256, 256) and sT.shape == (2, 256)
    # v[m, k] = fl32(D4(q) * s[k/128][m]) with numpy binary32 multiplies
    d = TAB[q].astype(np.float32)
    srow = np.repeat(s, 128, axis=0).T            # [M, K]: s[k/128][m]
    v = (d * srow).astype(np.float32)
    for k in (0, 1, 77, 128, 200, 255):
        for mb in range(2):
            sb, cb = brute_group(v[mb * 128:(mb + 1) * 128, k])
            assert sT[mb, k].view(np.uint32) == sb.view(np.uint32)
            assert np.array_equal(qT[k, mb * 128:(mb + 1) * 128], cb)


def test_requant_invariants_single_linear():
    c = wl.single_linear()
    for t in (c.x, c.dy):
        q, s = oracle.quant_act_1x128(wl.bf16_bits(t))
        qT, sT = oracle.requant_128x1(q, s)
        M, K = q.shape
        d = TAB[q].astype(np.float32)
        v = (d * np.repeat(s, 128, axis=0).T).astype(np.float32)
        vg = v.reshape(M // 128, 128, K)                    # [mb, i, k]
        amax = np.abs(vg).max(axis=1)                       # [mb, k]
        exp_s = np.where(amax == 0, np.float32(1), amax / np.float32(448)).astype(np.float32)
        assert np.array_equal(sT.view(np.uint32), exp_s.view(np.uint32))
        arg = np.abs(vg).argmax(axis=1)                     # [mb, k]
        qTg = qT.reshape(K, M // 128, 128)                  # [k, mb, i]
        top = np.take_along_axis(qTg, arg.T[..., None], axis=2)[..., 0]
        nz = (amax != 0).T
        assert ((top[nz] & 0x7F) == 0x7E).all()


def test_requant_of_representable_is_identity():
    """If every token block already spans +-448 with scale 1, requant is the transpose."""
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 0x7F, size=(256, 128)).astype(np.uint8)
    codes[::128, :] = 0x7E      # row 0 and 128: one element per column block at 448
    codes[:, 0] = 0x7E          # and one per 1x128 row group
    q, s = oracle.quant_act_1x128(to_bits(TAB[codes].astype(np.float32)))
    assert (s == 1).all()
    qT, sT = oracle.requant_128x1(q, s)
    assert (sT == 1).all() and np.array_equal(qT, codes.T)
