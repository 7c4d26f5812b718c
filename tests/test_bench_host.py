"""Host-side pieces of bench.py that need no GPU: the two-stage pipeline
closed form it models the dispatch ring with, the percentile summary and the
algorithmic byte counts behind the roofline."""
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
