"""Host-side pieces of bench.py that need no GPU: the two-stage pipeline
closed form it models the dispatch ring with, the percentile summary, the
algorithmic byte counts behind the roofline, the DRAM-traffic figure that
is reported only for the kernel sources it was captured on, and the peak
the fractions divide by."""
import os

import bench
from combine_movement_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pipeline_worked_example.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if "=" in line:
            k, v = (x.strip() for x in line.split("=", 1))
            vals[k] = float(v)
    return vals


def test_pipeline_closed_form_reproduces_the_worked_example():
    g = _golden()
    n = int(g["N"])
    assert bench.pipeline_time(n, g["t_load_us"], g["t_compute_us"]) == g["pipelined_us"]
    assert n * (g["t_load_us"] + g["t_compute_us"]) == g["serial_us"]
    assert bench.pipeline_time(0, 3.0, 5.0) == 0.0
    assert bench.pipeline_time(1, 3.0, 5.0) == 8.0   # one unit pays both stages


def test_spread_is_median_p10_p90_in_us():
    ms = [0.001 * (i + 1) for i in range(100)]     # 1 .. 100 µs
    med, p10, p90 = bench.spread(ms)
    assert abs(med - 50.5) < 1e-9 and p10 < 12 and p90 > 89


def test_algorithmic_bytes_of_the_deepseek_workload():
    wl = W.DEEPSEEK_PREFILL
    ab = bench.algorithmic_bytes(wl.T, wl.H, wl.K, wl.E, wl.T * wl.K)
    row = 2 * wl.H
    assert ab["dispatch"] == wl.T * row + wl.T * wl.K * row + 4 * wl.T * wl.K
    assert ab["combine"] == wl.T * wl.K * row + 8 * wl.T * wl.K + wl.T * row
    assert ab["dispatch"] == 528_613_376


def _tree_with_traffic(tmp_path):
    """A copy of the kernel sources and of the committed DRAM-traffic record
    under tmp_path, laid out as bench.py expects them under its root."""
    import json
    import shutil
    root = tmp_path / "root"
    shutil.copytree(os.path.join(bench.ROOT, "combine_movement_gb300", "csrc"),
                    root / "combine_movement_gb300" / "csrc")
    (root / "profiles").mkdir()
    shutil.copy(os.path.join(bench.ROOT, "profiles", "dram_traffic.json"),
                root / "profiles" / "dram_traffic.json")
    rec = json.load(open(root / "profiles" / "dram_traffic.json"))
    return root, rec


def test_kernel_traffic_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    """roofline.traffic comes from the committed ncu record while the
    kernel's sources hash to the recorded value, and is null once any of
    them changes."""
    root, rec = _tree_with_traffic(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    for kernel in ("dispatch", "combine"):
        # a record that matches the copied sources, whatever their state
        rec[kernel]["sources_sha256"] = bench.sources_sha256(rec[kernel]["sources"])
    import json
    json.dump(rec, open(root / "profiles" / "dram_traffic.json", "w"))
    assert bench.kernel_traffic("dispatch") == int(rec["dispatch"]["bytes_per_launch"])
    assert bench.kernel_traffic("combine") == int(rec["combine"]["bytes_per_launch"])
    # a header both kernels include changes: neither figure is reported
    shared = set(rec["dispatch"]["sources"]) & set(rec["combine"]["sources"])
    name = sorted(shared)[0]
    path = root / "combine_movement_gb300" / "csrc" / name
    path.write_text(path.read_text() + "\n// edited\n")
    assert bench.kernel_traffic("dispatch") is None
    assert bench.kernel_traffic("combine") is None
    assert bench.kernel_traffic("layout") is None  # no record at all


def test_peak_is_the_measured_copy_bandwidth_else_the_fallback(tmp_path, monkeypatch):
    import json
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    v, src = bench.peak_hbm()
    assert v == bench.FALLBACK_HBM_GBS and src.startswith("fallback")
    json.dump({"hbm_gbs": 6785.2}, open(tmp_path / "MEASURED_PEAKS.json", "w"))
    v, src = bench.peak_hbm()
    assert v == 6785.2 and src.startswith("measured")
