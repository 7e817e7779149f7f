"""The benchmark's reference arm runs on the CPU: the oracle as it stands, timed on whole decode
tokens, printed as one JSON line with the fields the comparison with the GPU arm needs (same
metric and unit, impl "reference", its own cpu_baseline and e2e).  Run here on the reduced
profiling case (4 layers, 2048-row lm_head) so that the CPU suite stays short."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "1",
                          "--layers", "4", "--vocab", "2048"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    import bench
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tok/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 2
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and "whole 4-layer tokens" in cb["sample"]
    assert abs(d["ms_per_step"] - 1e3 / d["value"]) <= 1e-6 * d["ms_per_step"]
    assert "REDUCED" in d["config"]["workload"]
    assert d["e2e"] == {"value": d["value"], "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
