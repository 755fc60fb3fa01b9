"""GPU parity of the FP8 KV cache (per-head scales recalibrated after a model
update, entries written with them) against the CPU oracle: scales and codes
bit-exact, called through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from fp8_block_quantized_gb300 import workloads as wl
from tests.gpu_util import assert_codes_equal, assert_scales_equal, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def jet(torch_cuda):
    import fp8_block_quantized_gb300 as j
    j.load()
    return j


def kv_batch(T, H, D, seed, spread=6.0):
    """K or V entries: N(0,1) with a per-head magnitude 2^U(-spread, spread) and
    a few outlier channels, BF16 [T, H, D]."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, H, D), generator=g)
    x *= torch.exp2((torch.rand((1, H, 1), generator=g) * 2 - 1) * spread)
    x[:, :, :: max(D // 8, 1)] *= 20.0
    return x.to(torch.bfloat16)


def check_calibrate(jet, x):
    s = jet.kv_calibrate(x.cuda())
    torch.cuda.synchronize()
    s_ref = oracle.kv_calibrate(bits(x))
    assert_scales_equal(s, s_ref, "kv scales")
    return s, s_ref


def check_write(jet, x, s, s_ref, slots, S, fill=0x55):
    T, H, D = x.shape
    cache = torch.full((S, H, D), fill, dtype=torch.uint8, device="cuda")
    jet.jet_kv_cache_write(x.cuda(), s, torch.from_numpy(slots).cuda(), cache)
    torch.cuda.synchronize()
    ref = np.full((S, H, D), fill, np.uint8)
    oracle.kv_cache_write(bits(x), s_ref, slots, ref)
    assert_codes_equal(cache, ref, "kv cache")


@pytest.mark.parametrize("T,H,D", [(1, 1, 16), (37, 8, 128), (300, 4, 64), (129, 2, 256), (64, 32, 128),
                                   (33, 3, 128), (50, 5, 16), (9, 24, 128)])
def test_calibrate_and_write(jet, T, H, D):
    x = kv_batch(T, H, D, seed=T * H + D)
    s, s_ref = check_calibrate(jet, x)
    rng = np.random.default_rng(T)
    S = 2 * T + 5
    slots = rng.permutation(S)[:T].astype(np.int64)
    check_write(jet, x, s, s_ref, slots, S)


def test_recalibrated_after_an_update(jet):
    """Scales from the batch before an update, then new scales from the
    batch after it; entries of both batches written with their own scales,
    later entries saturating where they exceed the older calibration."""
    T, H, D, S = 256, 8, 128, 1024
    a = kv_batch(T, H, D, seed=1)
    b = (kv_batch(T, H, D, seed=2).float() * 3).to(torch.bfloat16)   # the updated model
    sa, sa_ref = check_calibrate(jet, a)
    check_write(jet, b, sa, sa_ref, np.arange(T, dtype=np.int64), S)   # stale scales: saturation
    sb, sb_ref = check_calibrate(jet, b)
    check_write(jet, b, sb, sb_ref, np.arange(T, 2 * T, dtype=np.int64), S)


def test_edge_heads_and_slots(jet):
    T, H, D = 40, 6, 128
    x = kv_batch(T, H, D, seed=7).float()
    x[:, 1] = 0.0                          # an all-zero head: scale 1
    x[:, 2] *= 2.0 ** -100                 # a scale below 2^-90: the exact slow division
    x[:, 3, 5] = -0.0
    x[0, 4, :] = 3.3895e38                 # BF16 max in one entry
    x = x.to(torch.bfloat16)
    s, s_ref = check_calibrate(jet, x)
    slots = np.arange(T, dtype=np.int64)
    slots[3], slots[9] = -1, 10**12        # skipped
    check_write(jet, x, s, s_ref, slots, T)


def test_full_layer_prefill(jet):
    """One layer's keys for a 65536-token prefill of the 8B model (8 KV heads x 128)."""
    x = kv_batch(65536, 8, 128, seed=11)
    s, s_ref = check_calibrate(jet, x)
    slots = np.random.default_rng(0).permutation(65536 + 4096)[:65536].astype(np.int64)
    check_write(jet, x, s, s_ref, slots, 65536 + 4096)


def test_empty_batches(jet):
    e = torch.empty((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    s = jet.kv_calibrate(e)
    assert (s == 1.0).all()                # nothing calibrated: scale 1
    cache = torch.zeros((4, 8, 128), dtype=torch.uint8, device="cuda")
    jet.jet_kv_cache_write(e, s, torch.empty((0,), dtype=torch.int64, device="cuda"), cache)
    assert (cache == 0).all()
