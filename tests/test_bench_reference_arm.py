"""bench.py --impl reference (the oracle timed on the host cores) runs without
a GPU and prints one JSON line with the fields its contract names."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_prints_its_line():
    d = run("--impl", "reference", "--steps", "1", "--warmup", "1")
    assert d["impl"] == "reference" and d["data"] == "synthetic" and d["dtype"] == "f64"
    assert d["metric"] and d["unit"] == "GB/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 1 and d["n_gpus"] == 1 and d["vs_baseline"] is None
    assert d["config"]["workload"] == "llama8b_decode"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_takes_the_other_workloads():
    for w in ("tiny_decode", "prefix_sharing"):
        d = run("--impl", "reference", "--workload", w, "--steps", "1", "--warmup", "0")
        assert d["impl"] == "reference" and d["config"]["workload"] == w and d["value"] > 0
