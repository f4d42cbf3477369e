"""bench.py's reference arm runs on the host cores (the oracle), so its JSON line can be checked on a CPU host."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [x for x in res.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "llama3-8b-layer-N32768-k10pct" and d["config"]["k"] == 3277
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0


def test_traffic_record_is_tied_to_workload_and_code():
    # the committed DRAM-traffic capture is reported only for its workload and
    # for the code it was taken on (else null)
    sys.path.insert(0, ROOT)
    import bench
    from predicted_token_importance_tb_b300 import build
    with open(os.path.join(ROOT, "profiles", "fused_fast_traffic.json")) as f:
        rec = json.load(f)
    got = bench._traffic(rec["workload"])
    if build.code_hash(rec["code_units"]) == rec["code_hash"]:
        assert got == rec["dram_bytes_per_launch"]
    else:
        assert got is None
    assert bench._traffic("another-workload") is None
