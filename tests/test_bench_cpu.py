"""bench.py's host-side parts, on the CPU: the reference arm (the float64
oracle timed on the host cores) prints one JSON line with the fields the
measurement contract asks for, and the helpers that turn timings into
rates, ceilings and whole-job figures compute what they say."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_prints_one_contract_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True, env=env,
                         timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["steps"] == 1 and d["warmup"] >= 3 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["config"]["workload"] == "causal_fwdbwd_b8h12_n2048_d64"


def test_rate_and_ceiling_helpers():
    st = {"median": 2.0, "min": 1.0, "mean": 2.5, "n": 50}
    r = bench._rate(4e12, st, peak=1000.0)
    assert r["tflops"] == 2000.0 and r["tflops_best"] == 4000.0 and r["frac"] == 2.0
    assert r["launches"] == 50 and r["ms_median"] == 2.0 and r["ms_min"] == 1.0
    m = bench.mufu_ceiling(64, 2000.0, 100)
    # 32 exp2 per clock per SM x 100 SMs x 2 GHz = 6.4e12 exp2/s; x 4 d FLOPs = 1638.4 TFLOP/s
    assert m["fwd_tflops"] == pytest.approx(1638.4)
    assert m["bwd_tflops"] == pytest.approx(4096.0)
    s = bench._stats([3.0, 1.0, 2.0])
    assert s == {"median": 2.0, "min": 1.0, "mean": 2.0, "n": 3}


def test_whole_job_rate_and_window_pairs():
    # weak scaling: every rank's FLOPs in the slowest rank's time
    assert bench.whole_job_tflops(4, 1e12, 1.0) == pytest.approx(4000.0)
    # causal window of W keys over N queries: sum_i min(i + 1, W)
    N, W = 10, 3
    assert bench.window_pairs(N, W) == sum(min(i + 1, W) for i in range(N))
    assert bench.window_pairs(4, 10) == 4 * 5 // 2
