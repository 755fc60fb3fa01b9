"""Host-side logic of bench.py (no GPU): the roofline traffic lookup is keyed
by the kernels' source hash, and the CPU samples' work matches the
algorithmic counts the GPU arm uses."""
import json
import os

import pytest

import bench


def test_traffic_only_for_the_captured_source(tmp_path, monkeypatch):
    d = json.load(open(os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")))
    ent = d["train8b_layer_M8192"]["gemm_fp8_wgrad"]
    assert bench.measured_traffic("gemm_fp8_wgrad", "train8b_layer_M8192") in (ent["dram_bytes_per_launch"], None)
    # a hash that does not match the sources gives no traffic
    fake = {"train8b_layer_M8192": {"gemm_fp8_wgrad": dict(ent, sources_sha256_16="0" * 16)}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(fake))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("gemm_fp8_wgrad", "train8b_layer_M8192") is None
    assert bench.measured_traffic("gemm_fp8_fwd", "train8b_layer_M8192") is None


def test_source_hash_covers_every_listed_file():
    h1 = bench.source_hash(["gemm.cu"])
    h2 = bench.source_hash(["gemm.cu", "sm100_ptx.cuh"])
    assert len(h1) == 16 and h1 != h2


@pytest.mark.parametrize("workload,unit", [("train8b", "TFLOP/s"), ("sync", "GB/s"),
                                           ("kvcache", "GB/s"), ("moe", "TFLOP/s")])
def test_cpu_sample_units_and_work(workload, unit):
    smp = bench.CpuSample(workload)
    assert smp.unit == unit and smp.amount > 0 and smp.desc
    if workload == "train8b":
        assert smp.amount == 3 * 2 * 128 * 4096 * 4096     # q projection chain at 128 tokens
    assert smp.rate(2, 1.0) == pytest.approx(2 * smp.amount / (1e12 if unit == "TFLOP/s" else 1e9))


def test_job_rate_sums_ranks():
    assert bench.job_rate(4, 1e12, 1000.0, 1e12) == pytest.approx(4.0)
