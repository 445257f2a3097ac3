"""The benchmark's reference arm (the CPU oracle) run as a user runs it, on
CPU: one JSON line with the keys of the benchmark contract, the oracle's
arithmetic type, and an end-to-end figure with no host/device copies."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["steps"] == 1 and d["warmup"] >= 3          # the benchmark enforces three warm-up steps
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["dtype"] == "f64" and d["vs_baseline"] is None
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "8b_swiglu_q4_0_m2048"
    assert (d["config"]["M"], d["config"]["N"], d["config"]["K"]) == (2048, 14336, 4096)
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == d["value"] and cpu["cores"] >= 1 and cpu["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
