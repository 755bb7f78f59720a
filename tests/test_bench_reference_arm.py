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
    # the GPU arm's description of the same workload, word for word
    sys.path.insert(0, ROOT)
    import bench
    import workloads as wl
    assert d["config"]["workload"] == bench.decode_describe(wl.llama8b_decode(), True)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_takes_the_other_workloads():
    for w in ("tiny_decode", "prefix_sharing"):
        d = run("--impl", "reference", "--workload", w, "--steps", "1", "--warmup", "0")
        assert d["impl"] == "reference" and d["config"]["workload"].startswith(w + ":") and d["value"] > 0


def test_clock_summary_reads_the_timed_window():
    """The bench's nvidia-smi sampler: median SM clock over the timed window,
    the throttle reasons seen active in it, the nearest samples when none
    fall inside, and a marker when there are none at all."""
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler(0)

    def row(sm, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
        return f"0, {sm}, 2070, 900.5, 0x0, {hw}, {hwt}, {swt}, {cap}"

    c.samples = [(0.0, row(1200)), (1.0, row(2070)), (1.1, row(2040, cap="Active")), (1.2, row(2010)),
                 (5.0, row(900, hw="Active")), (6.0, "garbled")]
    s = c.summary(0.98, 1.22)
    assert s["sm_mhz"] == 2040 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]
    assert s["samples"] == 3 and s["window"] == "timed"
    s = c.summary(2.0, 3.0)                       # no sample inside: the last ones before its end
    assert s["window"] == "nearest" and s["samples"] == 4 and s["reasons"] == ["sw_power_cap"]
    s = c.summary(4.9, 5.1)
    assert s["reasons"] == ["hw_slowdown"] and s["sm_mhz"] == 900
    c.samples = []
    assert c.summary(0, 1)["reasons"] == ["no samples"]


def test_reference_arm_other_ranks_exit_quietly():
    """Under torchrun the reference arm runs on rank 0 alone; other ranks do no
    work, print nothing and exit 0."""
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and not r.stdout.strip()
