"""bench.py's output contract on a GPU, at the mid-size workload (N = 16,384,
H3 width): one JSON line with the metric, the device-timed value, the
roofline of the attention, the end-to-end legs with their byte counts, SM
clocks and host-link rates, the launch count, and the peak-memory record."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_on_the_mid_workload():
    steps = 3
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "mid", "--steps", str(steps),
                        "--warmup", "3", "--no-cpu-baseline", "--no-pack-record"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    n, C = 16384, 7168
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == 3
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    fl = 2 * n * C * 3 * C + 4 * n * n * C
    assert d["value"] > 0 and abs(d["value"] - fl / (d["ms_per_step"] * 1e-3) / 1e12) < 1e-6 * d["value"]
    assert d["config"]["n_tokens"] == n and d["config"]["hidden"] == C
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["unit"] == "TFLOP/s" and 0 < rf["frac"] < 1.5
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert d["gpu_launches"] == 2 * steps
    assert set(d["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == n * C * 2 and e["d2h_bytes_per_step"] == n * C * 2
    assert set(e["host_link"]) == {"h2d_gbs", "d2h_gbs"} and e["host_link"]["h2d_gbs"] > 0
    for leg in ("e2e_two_phase", "e2e_host_staged"):
        assert d[leg]["value"] > 0 and d[leg]["host_link"]["h2d_gbs"] > 0, leg
    assert 0 < d["peak_ratio"] <= 0.55
