"""The benchmark's reference arm (the fp64 oracle on the host cores) prints one
JSON line with the keys and types the benchmark contract fixes; it needs no GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_reference(*extra, env=None):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        *extra], capture_output=True, text=True, timeout=600, cwd=ROOT,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES="", **(env or {})))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_json_line():
    import bench
    d = run_reference("--steps", "2", "--warmup", "3")
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC
    assert d["unit"] == "GB/s (weight stream)" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["scaling"] == "weak" and d["vs_baseline"] is None and d["dtype"] == "f64"
    assert d["config"]["workload"] == "decode"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert "columns" in cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert d["gpu_launches"] == 0


def test_reference_arm_bounds_its_sample():
    """A heavy workload over many steps: the column (then row) sample shrinks so
    that the run stays within its time budget.  (One oracle thread: waking a
    team of threads costs milliseconds per call on some hosts, which would set
    a floor under the step that has nothing to do with the sampling.)"""
    d = run_reference("--workload", "prefill_sweep", "--steps", "100", "--warmup", "3",
                      "--ref-seconds", "10", env={"OMP_NUM_THREADS": "1"})
    assert d["steps"] == 100
    assert "columns" in d["cpu_baseline"]["sample"]
    assert d["ms_per_step"] * 100 / 1e3 < 20                   # the timed steps fit the budget


def test_reference_arm_under_torchrun_prints_once():
    """Launched like the multi-GPU bench (torchrun, two ranks; gloo here): rank 0
    alone runs the oracle and prints the line, the other rank exits 0."""
    r = subprocess.run(
        [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
         "--master-addr", "127.0.0.1", "--master-port", "29547",
         os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2", "--warmup", "3"],
        capture_output=True, text=True, timeout=600, cwd=ROOT,
        env=dict(os.environ, CUDA_VISIBLE_DEVICES="", W4A16_BENCH_BACKEND="gloo"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
