"""bench.py end to end on the GPU: one JSON line with the fields the
benchmark promises (metric, throughput, roofline of the dominant kernel,
end-to-end throughput with its copied bytes, clocks, launch count and the
oracle's CPU baseline), for the default decode workload and the mixed one."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "5",
                        "--warmup", "3", *args], capture_output=True, text=True, timeout=900,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def _common(d):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "dtype", "data", "config", "roofline", "e2e",
              "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["value"] > 0 and d["gpu_launches"] > 0
    r = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert 0 < r["frac"] < 2 and abs(r["achieved"] / r["peak"] - r["frac"]) < 1e-9
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]


def test_default_decode_line():
    d = _run("--cpu-sample-s", "0.5")
    _common(d)
    assert d["roofline"]["bound"] == "hbm" and d["roofline"]["unit"] == "GB/s"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    ca = d["cpu_baseline_all_cores"]
    assert ca["kind"] == "oracle" and ca["cores"] >= 1 and ca["value"] > 0 and ca["sample"]
    b = d["roofline"]["back_to_back"]
    assert b["ms_per_launch"] > 0 and abs(b["achieved"] / d["roofline"]["peak"] - b["frac"]) < 1e-9


@pytest.mark.parametrize("schedule", [(), ("--mixed-serial",)])
def test_mixed_step_line_reports_the_tensor_roofline(schedule):
    d = _run("--workload", "5", "--no-cpu-baseline", *schedule)
    _common(d)
    assert ("beside" in d["config"]["step_calls"]) == (not schedule)
    assert d["roofline"]["bound"] == "tensor" and d["roofline"]["unit"] == "TFLOP/s"
    assert d["decode_roofline"]["bound"] == "hbm"
    assert d["decode_roofline"]["back_to_back"]["ms_per_launch"] > 0
    assert d["tokens_per_s"] > 0
