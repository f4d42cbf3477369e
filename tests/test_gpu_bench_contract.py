"""bench.py's own arm on the GPU: one JSON line with every key of the contract, consistent with itself."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_bench_line_carries_every_key():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    res = subprocess.run([sys.executable, "bench.py", "--steps", "20", "--warmup", "3", "--no-e2e",
                          "--no-cpu-baseline"], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [x for x in res.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "clocks", "gpu_launches", "kernel_us",
                "median_of_5", "warm_l2"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] >= 3
    assert d["higher_is_better"] is True and d["value"] > 0
    # value is steps per second of the timed steps; kernel_us is the same time per step
    assert abs(d["value"] * d["ms_per_step"] / 1e3 - 1.0) < 1e-6
    assert abs(d["kernel_us"] - d["ms_per_step"] * 1e3) < 1e-6
    r = d["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in r, key
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9 and 0.0 < r["frac"] < 1.5
    # one decode-step kernel per timed step
    assert d["gpu_launches"] >= d["steps"]
    assert d["config"]["workload"] == "llama3-8b-layer-N32768-k10pct" and "l2_defeat" in d["config"]
    assert d["warm_l2"]["us_per_step"] > 0 and d["median_of_5"]["us_per_step"] > 0
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
