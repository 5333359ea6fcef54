"""bench.py's host logic on the CPU: the reference arm's JSON line (the oracle
timed on host cores) for a dense and a sparse workload, the clock-sample
filter, the sparse work count and the DRAM-traffic lookup. No GPU is
touched."""
import datetime
import json
import os
import subprocess
import sys

import torch

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run_reference(workload):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          workload, "--steps", "1", "--warmup", "0", "--ref-budget", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


def _check_reference_line(line, workload):
    assert line["impl"] == "reference"
    assert line["config"]["workload"] == workload
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]


def test_reference_arm_dense():
    _check_reference_line(_run_reference("tiny_s128_d64"), "tiny_s128_d64")


def test_reference_arm_sparse():
    line = _run_reference("csa_small_t512")
    _check_reference_line(line, "csa_small_t512")
    assert line["metric"] == bench.SPARSE_METRIC


def test_clock_samples_inside_the_timed_region_only(tmp_path):
    s = bench.ClockSampler(0)
    s.proc = object()  # a sampler that ran
    s.path = str(tmp_path / "clocks.csv")
    t0 = datetime.datetime(2026, 1, 1, 12, 0, 0)
    s.t_begin, s.t_end = t0 + datetime.timedelta(seconds=1), t0 + datetime.timedelta(seconds=3)
    rows = []
    for i, (mhz, cap) in enumerate([(1000, "Active"), (2000, "Not Active"), (1990, "Active"), (500, "Not Active")]):
        t = t0 + datetime.timedelta(seconds=i + 0.5)
        rows.append(f"{t.strftime('%Y/%m/%d %H:%M:%S.%f')[:-3]}, 0, {mhz}, 2070, 900.0, 0x0, Not Active, "
                    f"Not Active, Not Active, {cap}")
    (tmp_path / "clocks.csv").write_text("\n".join(rows) + "\n")
    summ = s.summary()
    assert summ["samples"] == 2                    # 1.5 s and 2.5 s fall inside [1 s, 3 s]
    assert summ["sm_mhz"] == 1995.0 and summ["sm_max_mhz"] == 2070.0
    assert summ["reasons"] == ["sw_power_cap"]


def test_sparse_work_counts_filled_slots():
    from attention_fwd_bwd_gb300.inputs import SPARSE_BY_NAME
    w = SPARSE_BY_NAME["csa_small_t512"]
    idx = torch.tensor([[[0, -1, 3, -1], [-1, -1, -1, -1]]], dtype=torch.int32)
    assert bench.sparse_flops(w, idx) == 2.0 * w.H * (w.DK + w.DV) * 2


def test_traffic_is_keyed_to_workload_and_kernel_sources(monkeypatch):
    """The roofline's DRAM traffic reads only for a workload with a capture
    taken on the current kernel sources: a different workload, or sources
    whose hash changed since, give None."""
    dense = bench.kernel_source_hash(bench.DENSE_SOURCES)
    sparse = bench.kernel_source_hash(bench.SPARSE_SOURCES)
    assert dense != sparse
    monkeypatch.setattr(bench, "TRAFFIC", {"w_dense": (dense, 1.5e9), "w_sparse": (sparse, 2.5e9),
                                           "w_stale": ("0" * 16, 3.5e9)})
    assert bench.traffic_for("w_dense", bench.DENSE_SOURCES) == 1.5e9
    assert bench.traffic_for("w_sparse", bench.SPARSE_SOURCES) == 2.5e9
    assert bench.traffic_for("w_sparse", bench.DENSE_SOURCES) is None
    assert bench.traffic_for("w_stale", bench.DENSE_SOURCES) is None
    assert bench.traffic_for("w_missing", bench.DENSE_SOURCES) is None
