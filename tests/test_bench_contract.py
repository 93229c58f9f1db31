"""The benchmark's reference arm runs on the CPU (the float64 oracle), so its
JSON line can be checked here: one line on stdout with the metric of the
GPU arm, its workload, and the cpu_baseline and e2e objects the contract asks
of the reference line."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "state-updates/s" and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] >= 3          # at least 3 warm-up steps, always
    assert d["n_gpus"] == 1 and d["scaling"] == "weak"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["vs_baseline"] is None                      # the pages publish no number
    assert d["config"]["B"] == 256 and d["config"]["H"] == 48 and d["config"]["HV"] == 96
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"] and cb["unit"] == d["unit"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
