"""bench.py's JSON line on small cases: the keys and their relations that the benchmark
contract fixes (metric, timing, roofline, end-to-end copies, launches, clocks).

Runs the script as a user would, in a subprocess, on the tiny workload, on the first 8
sequences of the INT8 batch and on one sequence of the long-context batch (both split
sequences into partitions, so the reduce kernel runs too).
The end-to-end leg checks its read-back output against the device path itself and
raises if they differ, which fails the run here.
"""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args):
    r = subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


@pytest.mark.parametrize("args", [
    ("--workload", "tiny"),
    ("--workload", "int8_cb", "--seqs", "8"),
    ("--workload", "long_32k", "--seqs", "1"),
])
def test_bench_line(args):
    d = _bench(*args, "--steps", "5", "--warmup", "3", "--no-cpu-baseline")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == args[1]

    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert r["launches_timed"] == 5
    assert 0 < r["median_launch_ms"] <= r["p90_launch_ms"]
    # the achieved rate is the algorithmic bytes over the mean launch
    assert abs(r["achieved"] - r["algorithmic_bytes_per_launch"] / (r["avg_launch_ms"] * 1e-3) / 1e9) \
        <= 5e-3 * r["achieved"] + 0.01  # both are rounded in the line

    e = d["e2e"]
    assert e["unit"] == "GB/s" and e["value"] > 0 and e["serial_value"] > 0
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0

    # every step launches at least the append and the decode kernel
    assert d["gpu_launches"] >= 2 * d["steps"]
    assert d["clocks"] is None or {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])  # None: no sample
