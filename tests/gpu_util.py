"""Helpers shared by the GPU parity tests (marshalling and comparisons only)."""
import numpy as np
import torch

from fp8_block_quantized_gb300 import workloads as wl


def to_dev(a, dtype=None):
    """numpy -> CUDA tensor (uint8 / float32 kept; uint16 BF16 bits -> bfloat16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def host(t):
    return t.detach().cpu().numpy()


def assert_codes_equal(q_gpu, q_ref, what="codes"):
    q = host(q_gpu)
    assert q.shape == q_ref.shape, (what, q.shape, q_ref.shape)
    bad = np.argwhere(q != q_ref)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first at {bad[:5].tolist()}: " \
        f"gpu {q[tuple(bad[0])]:#04x} oracle {q_ref[tuple(bad[0])]:#04x}"


def assert_scales_equal(s_gpu, s_ref, what="scales"):
    s = host(s_gpu).astype(np.float32)
    assert s.shape == s_ref.shape, (what, s.shape, s_ref.shape)
    bad = np.argwhere(s.view(np.uint32) != s_ref.astype(np.float32).view(np.uint32))
    assert bad.size == 0, f"{what}: {len(bad)} bitwise mismatches, first at {bad[:5].tolist()}: " \
        f"gpu {s[tuple(bad[0])]!r} oracle {s_ref[tuple(bad[0])]!r}"


def gemm_bound(ref):
    """|err| <= 2^-7 |ref| + 1e-3 * rms(ref row), elementwise."""
    rms = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
    return 2.0 ** -7 * np.abs(ref) + 1e-3 * rms


def assert_gemm_close(y_gpu, ref, what="gemm"):
    y = host(y_gpu.float()).astype(np.float64)
    assert y.shape == ref.shape, (what, y.shape, ref.shape)
    assert np.isfinite(y).all(), f"{what}: non-finite outputs"
    err = np.abs(y - ref)
    bound = gemm_bound(ref)
    bad = np.argwhere(err > bound)
    assert bad.size == 0, (f"{what}: {len(bad)} of {y.size} outside tolerance; first "
                           f"{bad[:3].tolist()}: gpu {y[tuple(bad[0])]!r} ref {ref[tuple(bad[0])]!r}")


def bits(t):
    return wl.bf16_bits(t)


def pair_tile_rows(M, seed=0):
    """Output rows that reach every 256-row pair tile in both of its 128-row
    halves (alternately the half's first row, its last row or a random one),
    plus the matrix's first and last rows.  Whole rows are compared, so each
    tile of the output is checked whatever order the tiles ran in."""
    rng = np.random.default_rng(1000 + seed)
    e = [0, M - 1]
    for t0 in range(0, M, 256):
        for h0 in (t0, t0 + 128):
            pick = (t0 // 256) % 3
            r = h0 if pick == 0 else h0 + 127 if pick == 1 else h0 + int(rng.integers(128))
            if r < M:
                e.append(r)
    return e
