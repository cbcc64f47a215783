"""Host logic of bench.py that its reported numbers depend on (no GPU).

* DRAM traffic is reported from a committed ncu summary only while that
  summary's recorded kernel-source hash matches the current sources.
* The per-launch distribution reports the median and the 10th/90th
  percentiles of the per-call times.
"""
from __future__ import annotations

import importlib.util
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test",
                                                  os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_traffic_needs_a_matching_hash(bench, tmp_path):
    good = bench.kernel_source_hash()
    prof = tmp_path / "p.md"
    prof.write_text(f"# x\n\nkernel_source_sha256_16: {good}\ntraffic_bytes_per_launch: 1234\n"
                    "other_traffic_bytes_per_launch: 99\n")
    assert bench.recorded_traffic(str(prof)) == 1234
    assert bench.recorded_traffic(str(prof), key="other_traffic_bytes_per_launch") == 99
    # A summary taken on other sources reports nothing.
    stale = "0" * 16 if good != "0" * 16 else "1" * 16
    prof.write_text(f"kernel_source_sha256_16: {stale}\ntraffic_bytes_per_launch: 1234\n")
    assert bench.recorded_traffic(str(prof)) is None
    # So does one without the key, or a missing file.
    prof.write_text(f"kernel_source_sha256_16: {good}\n")
    assert bench.recorded_traffic(str(prof)) is None
    assert bench.recorded_traffic(str(tmp_path / "absent.md")) is None
    # Keys count only at the start of a line (not inside prose).
    prof.write_text(f"see kernel_source_sha256_16: {good}\ntraffic_bytes_per_launch: 7\n")
    assert bench.recorded_traffic(str(prof)) is None


def test_source_hash_covers_every_listed_file(bench, tmp_path, monkeypatch):
    """Changing any listed source changes the hash."""
    csrc = tmp_path / "attention_attn_fwd_07_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cu").write_text("a")
    (csrc / "b.cuh").write_text("b")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash(["a.cu", "b.cuh"])
    (csrc / "b.cuh").write_text("b ")
    assert bench.kernel_source_hash(["a.cu", "b.cuh"]) != h0
    assert len(h0) == 16


def test_launch_stats(bench):
    t = list(np.arange(1, 101, dtype=np.float64))  # 1 .. 100 ms
    st = bench.launch_stats(t)
    assert st["n"] == 100
    assert st["median"] == pytest.approx(50.5)
    assert st["p10"] == pytest.approx(np.percentile(t, 10))
    assert st["p90"] == pytest.approx(np.percentile(t, 90))
    assert st["p10"] <= st["median"] <= st["p90"]


def test_summary_lists_every_line_last(bench):
    """The closing summary names the headline, each other workload, both
    decodes (MHA last, with its split count) and carries each line's own
    roofline fraction."""
    line = {"config": {"workload": "main"}, "value": 1600.0, "unit": "TFLOPS",
            "ms_per_step": 0.68, "roofline": {"frac": 0.86},
            "other_workloads": [
                {"workload": "d64", "value": 900.0, "metric": "TFLOPS", "ms_per_step": 0.04,
                 "roofline": {"frac": 0.48}},
                {"workload": "fp8", "value": 1700.0, "metric": "TFLOPS", "ms_per_step": 0.65,
                 "roofline": {"frac": 0.69}, "frac_of_bf16_peak": 0.92}],
            "decode_gqa": {"workload": "gqa", "value": 6900.0, "unit": "GB/s",
                           "ms_per_step": 0.31, "roofline": {"frac": 1.02}},
            "decode": {"workload": "mha", "value": 7100.0, "unit": "GB/s", "ms_per_step": 1.2,
                       "splits": 16, "roofline": {"frac": 1.05}}}
    s = bench.summary_of(line)
    assert [e[0] for e in s] == ["main", "d64", "fp8", "gqa", "mha, S=16"]
    assert [e[3] for e in s] == [0.86, 0.48, 0.69, 1.02, 1.05]
    assert s[-1][2] == "GB/s" and s[0][2] == "TFLOPS"
