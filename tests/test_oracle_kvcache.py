"""Pins for the oracle's FP8 KV cache (per-head scales recalibrated after a
model update, entries written with them).  They reduce it to the pinned 1x128
group rule, and check the codec's saturation and round trip, the monotone
calibration, and the slot scatter."""
import numpy as np

import oracle
from tests.test_oracle_swiglu import bf16


def tab():
    return oracle.e4m3_decode_table()


def test_one_token_of_128_channels_is_the_1x128_quantizer():
    rng = np.random.default_rng(1)
    H, D = 8, 128
    x = bf16(rng.standard_normal((1, H, D)) * np.exp2(rng.uniform(-8, 8, (1, H, 1))))
    s = oracle.kv_calibrate(x)
    cache = np.zeros((1, H, D), np.uint8)
    oracle.kv_cache_write(x, s, np.array([0]), cache)
    q_ref, s_ref = oracle.quant_act_1x128(x.reshape(H, D))
    assert np.array_equal(s.view(np.uint32), s_ref[0].view(np.uint32))
    assert np.array_equal(cache.reshape(H, D), q_ref)


def test_calibration_is_the_larger_of_two_batches_and_zero_gives_one():
    rng = np.random.default_rng(2)
    a = bf16(rng.standard_normal((50, 4, 64)))
    b = bf16(rng.standard_normal((70, 4, 64)) * 3)
    b[:, 2] = 0
    a[:, 3] = 0
    b[:, 3] = 0
    sa, sb = oracle.kv_calibrate(a), oracle.kv_calibrate(b)
    sab = oracle.kv_calibrate(np.concatenate([a, b]))
    assert np.array_equal(sab[:2], np.maximum(sa, sb)[:2])
    assert sab[2] == sa[2] and sb[2] == 1.0           # an all-zero batch has scale 1
    assert sab[3] == 1.0


def test_entries_beyond_the_calibrated_range_saturate():
    H, D = 2, 32
    calib = np.zeros((1, H, D), np.float32)
    calib[0, :, 0] = [448.0, 896.0]                   # scales 1 and 2
    s = oracle.kv_calibrate(bf16(calib))
    assert s.tolist() == [1.0, 2.0]
    x = np.zeros((1, H, D), np.float32)
    x[0, 0, :4] = [1000.0, -1000.0, 448.0, 464.0]
    x[0, 1, :3] = [1e4, -2.0, 0.5]
    cache = np.zeros((1, H, D), np.uint8)
    oracle.kv_cache_write(bf16(x), s, np.array([0]), cache)
    assert cache[0, 0, :4].tolist() == [0x7E, 0xFE, 0x7E, 0x7E]
    assert cache[0, 1, 0] == 0x7E and tab()[cache[0, 1, 1]] == -1.0 and tab()[cache[0, 1, 2]] == 0.25


def test_representable_entries_round_trip_at_scale_one():
    t = tab()
    vals = t[np.isfinite(t)].astype(np.float32)      # 254 values, |v| <= 448
    x = np.zeros((2, 1, 128), np.float32)
    x.reshape(-1)[:vals.size] = vals
    s = oracle.kv_calibrate(bf16(x))
    assert s[0] == 1.0
    cache = np.zeros((2, 1, 128), np.uint8)
    oracle.kv_cache_write(bf16(x), s, np.array([0, 1]), cache)
    got = t[cache.reshape(-1)[:vals.size]]
    assert np.array_equal(got, vals.astype(np.float64))


def test_slots_scatter_rows_and_skip_out_of_range():
    rng = np.random.default_rng(3)
    T, H, D, S = 6, 3, 64, 10
    x = bf16(rng.standard_normal((T, H, D)))
    s = oracle.kv_calibrate(x)
    dense = np.zeros((T, H, D), np.uint8)
    oracle.kv_cache_write(x, s, np.arange(T), dense)
    slots = np.array([7, 2, -1, 9, 10, 0])
    cache = np.full((S, H, D), 0x55, np.uint8)
    oracle.kv_cache_write(x, s, slots, cache)
    for t, sl in enumerate(slots):
        if 0 <= sl < S:
            assert np.array_equal(cache[sl], dense[t])
    untouched = [i for i in range(S) if i not in set(slots.tolist())]
    assert (cache[untouched] == 0x55).all()
