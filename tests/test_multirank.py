"""The N > 1 path of bench.py on CPU: two gloo ranks (replicas) agree on the
slowest rank's time and the whole-job rate (no GPU, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [6.0, 7.5][rank]                         # per-rank step times
        slowest = bench.max_over_ranks(ms, world, "cpu")
        rate = bench.job_rate(world, 10.72e12, slowest, 1e12)
        out.put((rank, slowest, rate))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_agree_on_max_time_and_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [7.5, 7.5]
    expected = 2 * 10.72e12 / 7.5e-3 / 1e12
    assert all(abs(r[2] - expected) < 1e-9 for r in res)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.job_rate(1, 2e12, 1000.0, 1e12) == pytest.approx(2.0)
