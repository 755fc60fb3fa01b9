"""Pins for the oracle's E4M3 codec (CPU only).

The codec is pinned against facts that do not come from the oracle itself:
the OCP E4M3FN landmarks, PyTorch's independent float8_e4m3fn conversion
(round-to-nearest-even, used only for |v| <= 448 where it does not saturate),
exhaustive round trips, and the neighbours of every rounding midpoint.
"""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def torch_decode_table():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def torch_encode(v):
    t = torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_decode_matches_torch_all_codes():
    ours = oracle.e4m3_decode_table()
    ref = torch_decode_table()
    nan_o, nan_r = np.isnan(ours), np.isnan(ref)
    assert (nan_o == nan_r).all()
    assert np.array_equal(ours[~nan_o], ref[~nan_r])
    # sign of zero
    assert math.copysign(1.0, ours[0x80]) == -1.0 and math.copysign(1.0, ours[0]) == 1.0


def test_decode_landmarks():
    d = oracle.e4m3_decode
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0          # max finite
    assert d(0x08) == 2.0 ** -6                            # min normal
    assert d(0x01) == 2.0 ** -9                            # min subnormal
    assert d(0x07) == 7 * 2.0 ** -9                        # max subnormal
    assert d(0x38) == 1.0
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))     # the only NaNs
    tab = oracle.e4m3_decode_table()
    assert np.isfinite(tab).sum() == 254
    pos = tab[:0x7F]
    assert (np.diff(pos) > 0).all(), "codes 0x00..0x7E must increase"


def test_round_trip_every_finite_code():
    tab = oracle.e4m3_decode_table()
    codes = np.array([c for c in range(256) if not np.isnan(tab[c])], np.uint8)
    vals = tab[codes].astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_midpoints_tie_to_even_and_neighbours():
    tab = oracle.e4m3_decode_table()
    for c in range(0x7E):
        lo, hi = tab[c], tab[c + 1]
        mid = np.float32((lo + hi) / 2)          # <= 5 significant bits: exact
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        got = oracle.e4m3_encode(np.array([mid, np.nextafter(mid, np.float32(0)),
                                           np.nextafter(mid, np.float32(1e9))],
                                          np.float32))
        assert got[0] == even, (hex(c), float(mid))
        assert got[1] == c and got[2] == c + 1
        # negative side: same code with the sign bit
        gotn = oracle.e4m3_encode(np.array([-mid], np.float32))
        assert gotn[0] == (even | 0x80)


def test_encode_matches_torch_random():
    rng = np.random.default_rng(1234)
    n = 200_000
    mag = np.exp2(rng.uniform(-14, math.log2(448), n)).astype(np.float32)
    v = (mag * rng.choice([-1, 1], n)).astype(np.float32)
    v = v[np.abs(v) <= 448]
    assert np.array_equal(oracle.e4m3_encode(v), torch_encode(v))


def test_saturation_and_zero_rules():
    e = lambda x: int(oracle.e4m3_encode(np.array([x], np.float32))[0])
    assert e(np.float32(448) * np.float32(1 + 2 ** -23)) == 0x7E
    assert e(464.0) == 0x7E and e(1e30) == 0x7E and e(-1e30) == 0xFE
    assert e(3.0e38) == 0x7E
    assert e(2.0 ** -10) == 0x00 and e(-(2.0 ** -10)) == 0x80
    assert e(1.5 * 2.0 ** -10) == 0x01
    assert e(0.0) == 0x00 and e(-0.0) == 0x80
    assert e(1e-45) == 0x00 and e(-1e-45) == 0x80          # binary32 subnormals


def test_sign_symmetry():
    rng = np.random.default_rng(7)
    v = rng.standard_normal(50_000).astype(np.float32) * 40
    assert np.array_equal(oracle.e4m3_encode(-v), oracle.e4m3_encode(v) ^ 0x80)


def test_worked_examples_codes():
    """Hand-derived codes (tests/golden/e4m3_worked_groups.txt), s = 1 group."""
    from tests.golden_io import load_worked_groups
    groups = load_worked_groups()
    a = groups["A"]
    vals = np.array([x for x, _ in a["entries"]], np.float32)
    want = np.array([c for _, c in a["entries"]], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(vals), want)
