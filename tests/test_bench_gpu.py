"""bench.py's own arm on the GPU: one short run (``--no-extras``: the timed
step alone, without the end-to-end loop, the oracle baseline and the other
legs) prints one JSON line that carries the contract's core fields, with
values that are consistent with each other (whole-job rate from the step
time, the roofline fraction from achieved over peak, this library's kernels
counted, the clocks sampled)."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_contract():
    pytest.importorskip("torch")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3",
                          "--no-extras"], capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] >= 3 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "causal_fwdbwd_b8h12_n2048_d64"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    # whole-job TFLOP/s from the step time: forward 4 B H N^2 d / 2 plus 2.5 times that backward
    flops = 3.5 * 4 * 8 * 12 * 2048 ** 2 * 64 / 2
    assert abs(d["value"] - flops / (d["ms_per_step"] * 1e-3) / 1e12) <= 0.01 * d["value"]
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) <= 1e-3
    assert d["gpu_launches"] >= 4 * d["steps"]  # forward, preprocess, main, finish per step
    c = d["clocks"]
    assert "sm_mhz" in c and "reasons" in c
