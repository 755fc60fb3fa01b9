"""bench.py's reference arm (the CPU oracle on a bounded sample of each
workload) on CPU: one JSON line with the contract's keys, in the unit of the
workload's GPU arm, and the same `config.workload` name."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("workload,unit", [("metric", "GB/s"), ("kvcache", "GB/s"),
                                           ("rollout", "TFLOP/s")])
def test_reference_line(workload, unit):
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", workload,
                        "--steps", "1", "--warmup", "0"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    assert line["impl"] == "reference" and line["unit"] == unit and line["value"] > 0
    for key in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "cpu_baseline", "e2e", "config"):
        assert key in line
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    import bench
    args = type("A", (), {"workload": workload, "tokens": 2048})()
    assert line["config"]["workload"] == bench.workload_name(args)


def test_reference_other_ranks_exit_without_work():
    """Under torchrun only rank 0 runs the reference arm; the others exit 0
    and print nothing."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "metric",
                        "--steps", "1"], cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]
