"""Throughput of exact attention (forward + backward) on GB300.

One step is one pass of the whole hot path over one batch: the forward
(fa_fwd) and the three backward stages (fa_bwd preprocess, main, finish) on
the causal forward+backward workload B=8, H=12, N=2048, d=64 with iid N(0,1)
bf16 inputs. The metric is TFLOP/s with the method's algorithmic count,
4 B H N^2 d for the forward (halved when causal) and 2.5x that for the
backward, and its fraction of the measured dense BF16 tensor peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: W untimed warm-up steps, then K steps between a barrier and a device
synchronisation on both sides, each step bracketed by CUDA events on the
stream the kernels run on; L2 is flushed (a 256 MiB write) between steps,
outside the events. Under torchrun every rank runs its own batch (weak
scaling; no collective in the data path) and rank 0 prints one JSON line
with the slowest rank's time.

``--impl reference`` times the float64 CPU oracle instead, on a bounded
sample of the same workload per step (rank 0 only).
"""

from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic_inputs as si  # noqa: E402

METRIC = "attention fwd/bwd TFLOP/s on 1 GB300 and % of dense BF16 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_PEAK_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=si.WORKLOADS[4].name)
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the end-to-end, CPU-baseline and long-forward legs")
    ap.add_argument("--only", default=None,
                    help="run one extra leg alone and print its JSON (for profiling): configs, "
                         "sweep, d256, decode, window, headsize, dropout, or workload:<name>")
    ap.add_argument("--decode-nk", type=int, default=32768,
                    help="cached keys per sequence in the decode leg")
    ap.add_argument("--sweep-n", default="4096,8192,16384",
                    help="sequence lengths of the d=128 sweep (comma-separated)")
    ap.add_argument("--sweep-causal", choices=["both", "causal", "noncausal"], default="both")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0.0)), "measured"
    except Exception:
        return FALLBACK_PEAK_TFLOPS, 1700.0, "fallback"


def measured_hbm_gbs():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def window_pairs(N, window):
    """Visible (query, key) pairs of one head under a causal window."""
    w = min(window, N)
    return w * (w + 1) // 2 + (N - w) * w


def time_calls(fn, reps, warmup, stream, flush=None):
    """Median ms of fn() over `reps` launches on `stream` (CUDA events)."""
    return time_segments([fn], reps, warmup, stream, flush)[0]["median"]


def _stats(ts):
    import statistics
    return {"median": statistics.median(ts), "min": min(ts), "mean": sum(ts) / len(ts), "n": len(ts)}


def time_segments(fns, reps, warmup, stream, flush=None):
    """Per-call ms statistics of a sequence of launches: each rep flushes L2
    (outside the events), then runs fns[0], fns[1], ... on `stream` with a
    CUDA event between consecutive calls. Returns one statistics dict
    (median, min, mean, n) per call and one for the whole sequence."""
    import torch
    with torch.cuda.stream(stream):  # the flush runs on the timed stream, ahead of the calls
        for _ in range(warmup):
            if flush is not None:
                flush()
            for f in fns:
                f()
        torch.cuda.synchronize()
        mk = lambda: torch.cuda.Event(enable_timing=True)
        evs = [[mk() for _ in range(len(fns) + 1)] for _ in range(reps)]
        for e in evs:
            if flush is not None:
                flush()
            e[0].record(stream)
            for i, f in enumerate(fns):
                f()
                e[i + 1].record(stream)
        torch.cuda.synchronize()
    per = [_stats([e[i].elapsed_time(e[i + 1]) for e in evs]) for i in range(len(fns))]
    per.append(_stats([e[0].elapsed_time(e[-1]) for e in evs]))
    return per


def decode_leg(dev, stream, reps=20, Nk=32768):
    """Split-key-range decode: 8 sequences x 32 heads, one query over Nk
    (32768) cached keys (d = 128, causal). HBM-bound: every key and value is
    read once; the roofline counts K, V, Q, O and the fp32 partial states."""
    import torch
    import exact_io_aware_33_gb300 as fa
    B, H, Nq, d = 8, 32, 1, 128
    # drawn on the device (seeded): 2 x 1 G values would take long on the host
    g = torch.Generator(device=dev).manual_seed(4242)
    q = torch.randn(B, H, Nq, d, generator=g, device=dev).to(torch.bfloat16)
    k = torch.randn(B, H, Nk, d, generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn(B, H, Nk, d, generator=g, device=dev).to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, Nq, dtype=torch.float32, device=dev)
    splits = fa.fa_decode_num_splits(B, H, Nq, Nk, 0)
    ws = torch.empty(fa.fa_decode_workspace_bytes(B, H, Nq, Nk, d, 0), dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        ms = time_calls(lambda: fa.fa_decode_splitkv(q, k, v, causal=True, n_splits=0, out=o, lse=lse,
                                                     workspace=ws, stream=stream), reps, 3, stream)
    part = splits * B * H * Nq * (d + 1) * 4
    algo = 2 * B * H * Nk * d * 2 + 2 * B * H * Nq * d * 2 + B * H * Nq * 4 + 2 * part
    peak, src = measured_hbm_gbs()
    gbs = algo / (ms * 1e-3) / 1e9
    return {"workload": f"decode_b8h32_nq1_nk{Nk}_d128_causal", "splits": splits, "ms": round(ms, 4),
            "bytes": algo, "gbs": round(gbs, 1), "peak_gbs": peak, "frac": round(gbs / peak, 4),
            "bound": "hbm", "peak_source": f"{src} copy bandwidth (MEASURED_PEAKS.json)",
            "l2": f"inputs ({2 * B * H * Nk * d * 2 / 1e9:.1f} GB) larger than L2"}


def headsize_leg(dev, stream, flush, reps=10):
    """Queries/keys of head size 128 with values of head size 64 (causal,
    B=4 H=16 N=4096): forward and full backward. FLOPs per visible pair:
    2 (d + d_v) forward; 2 (3 d + 2 d_v) backward (S, dP, dV, dK, dQ)."""
    import torch
    import exact_io_aware_33_gb300 as fa
    B, H, N, d, dv = 4, 16, 4096, 128, 64
    g = torch.Generator(device="cpu").manual_seed(91)
    q, k = (torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).to(dev) for _ in range(2))
    v, do = (torch.randn(B, H, N, dv, generator=g).to(torch.bfloat16).to(dev) for _ in range(2))
    o = torch.empty(B, H, N, dv, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, H, N, dtype=torch.float32, device=dev)
    dq, dk, dvv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        ms_f = time_calls(lambda: fa.fa_fwd_ex(q, k, v, causal=True, out=o, lse=lse, stream=stream),
                          reps, 3, stream, flush)
        ms_b = time_calls(lambda: fa.fa_bwd_ex(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk,
                                               dv=dvv, workspace=ws, stream=stream),
                          reps, 3, stream, flush)
    pairs = B * H * N * (N + 1) / 2
    return {"workload": "headsize_causal_b4h16_n4096_d128_dv64", "fwd_ms": round(ms_f, 4),
            "fwd_tflops": round(2.0 * (d + dv) * pairs / (ms_f * 1e-3) / 1e12, 1),
            "bwd_ms": round(ms_b, 4),
            "bwd_tflops": round(2.0 * (3 * d + 2 * dv) * pairs / (ms_b * 1e-3) / 1e12, 1),
            "note": "backward = preprocess + main + finish"}


def window_leg(dev, stream, flush, reps=10):
    """Causal sliding window W = 1024 on B=1 H=16 N=8192 d=128: forward and
    backward; FLOPs count visible pairs only (4 d per pair forward, 2.5x
    that backward)."""
    import torch
    import exact_io_aware_33_gb300 as fa
    B, H, N, d, W = 1, 16, 8192, 128, 1024
    x = si.make_small(B, H, N, d, seed=77, with_grad=True)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        ms_f = time_calls(lambda: fa.fa_fwd_ex(q, k, v, causal=True, window=W, out=o, lse=lse,
                                               stream=stream), reps, 3, stream, flush)
        ms_b = time_calls(lambda: fa.fa_bwd_ex(q, k, v, o, lse, do, causal=True, window=W, dq=dq,
                                               dk=dk, dv=dv, workspace=ws, stream=stream),
                          reps, 3, stream, flush)
    f_fwd = 4.0 * d * B * H * window_pairs(N, W)
    return {"workload": "window_causal_b1h16_n8192_d128_w1024", "fwd_ms": round(ms_f, 4),
            "fwd_tflops": round(f_fwd / (ms_f * 1e-3) / 1e12, 1), "bwd_ms": round(ms_b, 4),
            "bwd_tflops": round(2.5 * f_fwd / (ms_b * 1e-3) / 1e12, 1),
            "note": "backward = preprocess + main + finish"}


def dropout_leg(dev, stream, flush, reps=10):
    """Dropout p = 0.1 on the forward+backward workload's shape (causal,
    B=8 H=12 N=2048 d=64): forward and full backward with the keep mask
    regenerated in both; FLOPs as without dropout (4 B H N^2 d / 2 forward,
    2.5x that backward), the generator's integer work not counted."""
    import torch
    import exact_io_aware_33_gb300 as fa
    w = si.workload("causal_fwdbwd_b8h12_n2048_d64")
    x = si.make_inputs(w, with_grad=True)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)
    p, seed = 0.1, 2024
    with torch.cuda.stream(stream):
        ms_f = time_calls(lambda: fa.fa_fwd_dropout(q, k, v, p, seed, 1, causal=True, scale=w.scale,
                                                    out=o, lse=lse, stream=stream), reps, 3, stream, flush)
        ms_b = time_calls(lambda: fa.fa_bwd_dropout(q, k, v, o, lse, do, p, seed, 1, causal=True,
                                                    scale=w.scale, dq=dq, dk=dk, dv=dv, workspace=ws,
                                                    stream=stream), reps, 3, stream, flush)
    f_fwd, f_bwd = step_flops(w)
    return {"workload": "dropout_p0.1_" + w.name, "fwd_ms": round(ms_f, 4),
            "fwd_tflops": round(f_fwd / (ms_f * 1e-3) / 1e12, 1), "bwd_ms": round(ms_b, 4),
            "bwd_tflops": round(f_bwd / (ms_b * 1e-3) / 1e12, 1),
            "step_tflops": round((f_fwd + f_bwd) / ((ms_f + ms_b) * 1e-3) / 1e12, 1),
            "note": "backward = preprocess + main + finish; keep mask from Philox4x32-10 in both"}


class AbiProblem:
    """Device buffers and C-ABI launches of one square problem [B, H, N, d]
    (N queries = N keys, d = d_v): the forward and the three backward stages."""

    def __init__(self, lib, x, causal, scale):
        import torch
        self.lib, self.x, self.causal, self.scale = lib, x, 1 if causal else 0, scale
        self.B, self.H, self.N, self.d = (int(n) for n in x["q"].shape)
        dev = x["q"].device
        self.o = torch.empty_like(x["q"])
        self.lse = torch.empty(self.B, self.H, self.N, dtype=torch.float32, device=dev)
        if "do" in x:
            self.dq, self.dk, self.dv = (torch.empty_like(x["q"]) for _ in range(3))
            self.ws_bytes = lib.fa_bwd_workspace_bytes(self.B, self.H, self.N, self.d)
            self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)

    @staticmethod
    def _p(t):
        return ctypes.c_void_p(t.data_ptr())

    def _ok(self, rc, what):
        if rc != 0:
            raise RuntimeError(f"{what}: {rc}")

    def fwd(self, stream):
        p, x = self._p, self.x
        self._ok(self.lib.fa_fwd_stream(p(x["q"]), p(x["k"]), p(x["v"]), p(self.o), p(self.lse),
                                        self.B, self.H, self.N, self.d, self.causal, self.scale,
                                        ctypes.c_void_p(stream.cuda_stream)), "fa_fwd_stream")

    def pre(self, stream):
        p = self._p
        self._ok(self.lib.fa_bwd_preprocess_stream(p(self.o), p(self.lse), p(self.x["do"]), self.B,
                                                   self.H, self.N, self.d, p(self.ws),
                                                   ctypes.c_size_t(self.ws_bytes),
                                                   ctypes.c_void_p(stream.cuda_stream)), "preprocess")

    def main(self, stream):
        p, x = self._p, self.x
        self._ok(self.lib.fa_bwd_main_stream(p(x["q"]), p(x["k"]), p(x["v"]), p(x["do"]), p(self.dk),
                                             p(self.dv), self.B, self.H, self.N, self.d, self.causal,
                                             self.scale, p(self.ws), ctypes.c_size_t(self.ws_bytes),
                                             ctypes.c_void_p(stream.cuda_stream)), "main")

    def post(self, stream):
        self._ok(self.lib.fa_bwd_finish_stream(self._p(self.dq), self.B, self.H, self.N, self.d,
                                               self._p(self.ws), ctypes.c_size_t(self.ws_bytes),
                                               ctypes.c_void_p(stream.cuda_stream)), "finish")


def _rate(flops, st, peak):
    """TFLOP/s at the median and the best launch, and the median's fraction of peak."""
    tf = flops / (st["median"] * 1e-3) / 1e12
    return {"ms_median": round(st["median"], 4), "ms_min": round(st["min"], 4), "launches": st["n"],
            "tflops": round(tf, 1), "tflops_best": round(flops / (st["min"] * 1e-3) / 1e12, 1),
            "frac": round(tf / peak, 4)}


def mufu_ceiling(d, sm_mhz, sms):
    """TFLOP/s the exponential unit allows: one exp2 per score element at 32
    per clock per SM (measured on GB300), against 4 d FLOPs per element in the
    forward (QK^T and PV) and 10 d in the backward (five contractions, one
    recomputed exponential)."""
    ex2_per_s = 32.0 * sms * sm_mhz * 1e6
    return {"ex2_per_clk_per_sm": 32, "sm_mhz": sm_mhz, "sms": sms,
            "fwd_tflops": round(ex2_per_s * 4 * d / 1e12, 1),
            "bwd_tflops": round(ex2_per_s * 10 * d / 1e12, 1)}


def config_legs(lib, dev, stream, flush, peak, sm_mhz, sms, reps=50, warmup=10, names=None):
    """Every named workload (or those in `names`), per pass: the forward, and
    where the workload has a backward the whole backward and its main kernel
    alone; the median and the best of `reps` launches, L2 flushed before each."""
    import exact_io_aware_33_gb300 as fa
    out = []
    for w in si.WORKLOADS:
        if names is not None and w.name not in names:
            continue
        x = {n: t.to(dev) for n, t in si.make_inputs(w, with_grad=w.backward).items()}
        pr = AbiProblem(lib, x, w.causal, w.scale)
        f_fwd = fa.flops_fwd(w.B, w.H, w.N, w.d, w.causal)
        mufu = mufu_ceiling(w.d, sm_mhz, sms)
        st = time_segments([lambda: pr.fwd(stream)], reps, warmup, stream, flush)
        out.append({"workload": w.name, "pass": "forward", **_rate(f_fwd, st[0], peak),
                    "mufu_ceiling_tflops": mufu["fwd_tflops"]})
        if w.backward:
            pr.fwd(stream)
            f_bwd = 2.5 * f_fwd
            st = time_segments([lambda: pr.pre(stream), lambda: pr.main(stream), lambda: pr.post(stream)],
                               reps, warmup, stream, flush)
            out.append({"workload": w.name, "pass": "backward (preprocess + main + finish)",
                        **_rate(f_bwd, st[3], peak), "mufu_ceiling_tflops": mufu["bwd_tflops"]})
            out.append({"workload": w.name, "pass": "backward main kernel", **_rate(f_bwd, st[1], peak),
                        "mufu_ceiling_tflops": mufu["bwd_tflops"]})
        del pr, x
    return out


def sweep_leg(lib, dev, stream, flush, peak, sm_mhz, sms, reps=50, warmup=10,
              lengths=(4096, 8192, 16384), masks=(True, False)):
    """d = 128 at N = 4096, 8192 and 16384, causal and non-causal, with
    B H N = 2^18 query rows at every N (1024 forward CTAs of 256 query rows:
    6.7 waves over 152 SMs): forward, whole backward and backward main kernel.
    Inputs: one seeded draw of iid N(0,1) bf16 rows, viewed as [B, H, N, 128]."""
    import exact_io_aware_33_gb300 as fa
    d, rows = 128, 1 << 18
    x0 = si.make_small(1, 1, rows, d, seed=4096, with_grad=True)
    x0 = {n: t.to(dev) for n, t in x0.items()}
    out = []
    for N in lengths:
        H = 16
        B = rows // (H * N)
        x = {n: t.view(B, H, N, d) for n, t in x0.items()}
        for causal in masks:
            pr = AbiProblem(lib, x, causal, 1.0 / math.sqrt(d))
            f_fwd = fa.flops_fwd(B, H, N, d, causal)
            st_f = time_segments([lambda: pr.fwd(stream)], reps, warmup, stream, flush)
            pr.fwd(stream)
            st_b = time_segments([lambda: pr.pre(stream), lambda: pr.main(stream), lambda: pr.post(stream)],
                                 reps, warmup, stream, flush)
            out.append({"B": B, "H": H, "N": N, "d": d, "causal": causal,
                        "fwd_ctas": B * H * ((N + 255) // 256),
                        "fwd": _rate(f_fwd, st_f[0], peak),
                        "bwd": _rate(2.5 * f_fwd, st_b[3], peak),
                        "bwd_main": _rate(2.5 * f_fwd, st_b[1], peak)})
            del pr
    mufu = mufu_ceiling(d, sm_mhz, sms)
    return {"points": out, "target_frac_fwd": 0.60,
            "min_fwd_frac": min(r["fwd"]["frac"] for r in out),
            "mufu_ceiling_tflops": {"fwd": mufu["fwd_tflops"], "bwd": mufu["bwd_tflops"]},
            "timing": f"median and best of {reps} launches after {warmup} warm-ups, L2 flushed before each"}


def d256_leg(lib, dev, stream, flush, peak, sm_mhz, sms, reps=50, warmup=10):
    """Head size d = d_v = 256 (forward only: B=2 H=16 N=4096, causal and
    non-causal; one 128-row query tile per CTA, 1024 CTAs)."""
    import exact_io_aware_33_gb300 as fa
    B, H, N, d = 2, 16, 4096, 256
    x = {n: t.to(dev) for n, t in si.make_small(B, H, N, d, seed=256, with_grad=False).items()}
    out = []
    for causal in (True, False):
        pr = AbiProblem(lib, x, causal, 1.0 / math.sqrt(d))
        st = time_segments([lambda: pr.fwd(stream)], reps, warmup, stream, flush)
        out.append({"B": B, "H": H, "N": N, "d": d, "causal": causal,
                    "fwd": _rate(fa.flops_fwd(B, H, N, d, causal), st[0], peak)})
        del pr
    return {"points": out, "mufu_ceiling_tflops": mufu_ceiling(d, sm_mhz, sms)["fwd_tflops"]}


def max_over_ranks(values, device, world):
    """Element-wise maximum of per-rank floats (the slowest rank's times)."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_tflops(world, flops_per_rank_step, ms_per_step):
    """Weak scaling: every rank processes its own batch in the slowest rank's time."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def rank_seed_offset(rank):
    """Each rank draws its own batch: the workload's seed plus the rank."""
    return rank


def step_flops(w):
    import exact_io_aware_33_gb300 as fa
    f = fa.flops_fwd(w.B, w.H, w.N, w.d, w.causal)
    return f, (fa.flops_bwd(w.B, w.H, w.N, w.d, w.causal) if w.backward else 0.0)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, every 200 ms."""

    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id):
        self.bus_id = (bus_id or "").lower()
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            if self.bus_id and parts[1].lower() != self.bus_id:
                continue
            rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(r[2]) for r in rows]
        busy = [s for s in sm if s > 0]
        sm_max = max(num(r[3]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        busy.sort()
        return {"sm_mhz": busy[len(busy) // 2] if busy else None, "sm_max_mhz": sm_max,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(num(r[4]) for r in rows)}


# ------------------------------------------------------------------ GPU arm
class Runner:
    """Buffers and C-ABI calls of one forward+backward step."""

    def __init__(self, w, device, seed_offset=0):
        import torch
        import exact_io_aware_33_gb300 as fa
        self.torch, self.fa, self.w, self.dev = torch, fa, w, device
        self.lib = fa.load_library()
        x = si.make_small(w.B, w.H, w.N, w.d, seed=w.seed + seed_offset, k_mult=w.k_mult,
                          with_grad=w.backward)
        self.host = x
        self.x = {k: t.to(device) for k, t in x.items()}
        self.o = torch.empty_like(self.x["q"])
        self.lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=device)
        if w.backward:
            self.dq = torch.empty_like(self.x["q"])
            self.dk = torch.empty_like(self.x["q"])
            self.dv = torch.empty_like(self.x["q"])
            self.ws_bytes = self.lib.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d)
            self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self.flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.launches_per_step = 4 if w.backward else 1

    def _p(self, t):
        return ctypes.c_void_p(t.data_ptr())

    def step(self, stream, ev=None):
        """Launch one step on `stream`; ev = dict of event pairs to record
        around the forward ("fwd") and the backward main kernel ("bwd_main"),
        either or both."""
        w, lib, p, x = self.w, self.lib, self._p, self.x
        ev = ev or {}
        sh = ctypes.c_void_p(stream.cuda_stream)
        c = 1 if w.causal else 0
        if "fwd" in ev:
            ev["fwd"][0].record(stream)
        rc = lib.fa_fwd_stream(p(x["q"]), p(x["k"]), p(x["v"]), p(self.o), p(self.lse),
                               w.B, w.H, w.N, w.d, c, w.scale, sh)
        if "fwd" in ev:
            ev["fwd"][1].record(stream)
        if rc != 0:
            raise RuntimeError(f"fa_fwd_stream: {rc}")
        if not w.backward:
            return
        wsb = ctypes.c_size_t(self.ws_bytes)
        rc = lib.fa_bwd_preprocess_stream(p(self.o), p(self.lse), p(x["do"]), w.B, w.H, w.N, w.d,
                                          p(self.ws), wsb, sh)
        if "bwd_main" in ev:
            ev["bwd_main"][0].record(stream)
        rc = rc or lib.fa_bwd_main_stream(p(x["q"]), p(x["k"]), p(x["v"]), p(x["do"]), p(self.dk),
                                          p(self.dv), w.B, w.H, w.N, w.d, c, w.scale, p(self.ws),
                                          wsb, sh)
        if "bwd_main" in ev:
            ev["bwd_main"][1].record(stream)
        rc = rc or lib.fa_bwd_finish_stream(p(self.dq), w.B, w.H, w.N, w.d, p(self.ws), wsb, sh)
        if rc != 0:
            raise RuntimeError(f"fa_bwd stages: {rc}")

    def flush_l2(self):
        self.flush_buf.zero_()


def timed_loop(runner, steps, warmup, barrier, stream, soak_s=0.0):
    """W warm-up steps, an optional untimed soak of about `soak_s` seconds of
    the same step (so that clocks sampled around the timed region reflect
    sustained load), then `steps` steps timed with CUDA events."""
    torch = runner.torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            runner.flush_l2()
            runner.step(stream)
    torch.cuda.synchronize()
    if soak_s > 0:
        t_end = time.perf_counter() + soak_s
        with torch.cuda.stream(stream):
            while time.perf_counter() < t_end:
                for _ in range(50):
                    runner.flush_l2()
                    runner.step(stream)
                torch.cuda.synchronize()
    mk = lambda: torch.cuda.Event(enable_timing=True)
    # Events around the dominant kernel only: an event recorded between two
    # kernels makes the second wait for the first to drain (about 3 us per
    # boundary at this size), so the step carries no others.
    dom = "bwd_main" if runner.w.backward else "fwd"
    evs = [{"step": (mk(), mk()), dom: (mk(), mk())} for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for e in evs:
            runner.flush_l2()
            e["step"][0].record(stream)
            runner.step(stream, e)
            e["step"][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - t0
    t = {k: [e[k][0].elapsed_time(e[k][1]) for e in evs] for k in ("step", dom)}
    return t, wall


def e2e_loop(runners, steps, warmup, stream):
    """The step through host buffers: every step copies its inputs from
    pinned host memory and every output back. Two device buffer sets and
    three streams (host-to-device copies, compute, device-to-host copies)
    let step i+1's upload and step i-1's download overlap step i's
    compute; the timed region runs from the first upload to the last
    download."""
    torch = runners[0].torch
    w = runners[0].w
    names_in = ["q", "k", "v"] + (["do"] if w.backward else [])
    h_in = {n: runners[0].host[n].pin_memory() for n in names_in}

    def outs(r):
        return [r.o, r.lse] + ([r.dq, r.dk, r.dv] if w.backward else [])

    h_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs(r)] for r in runners]
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])
    s_up, s_down = torch.cuda.Stream(), torch.cuda.Stream()
    mk = lambda: torch.cuda.Event(enable_timing=False)
    ev_in = [mk(), mk()]
    ev_comp = [mk(), mk()]
    ev_out = [mk(), mk()]
    used = [False, False]

    def one(i):
        b = i % 2
        r = runners[b]
        if used[b]:  # the buffer set's previous step has finished with its inputs and outputs
            s_up.wait_event(ev_comp[b])
            stream.wait_event(ev_out[b])
        with torch.cuda.stream(s_up):
            for n in names_in:
                r.x[n].copy_(h_in[n], non_blocking=True)
            ev_in[b].record(s_up)
        stream.wait_event(ev_in[b])
        r.step(stream)
        ev_comp[b].record(stream)
        s_down.wait_event(ev_comp[b])
        with torch.cuda.stream(s_down):
            for d, h in zip(outs(r), h_out[b]):
                h.copy_(d, non_blocking=True)
            ev_out[b].record(s_down)
        used[b] = True

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_up)
    for i in range(steps):
        one(warmup + i)
    z.record(s_down)
    torch.cuda.synchronize()
    return a.elapsed_time(z) / steps, h2d, d2h


def traffic_from_profiles(kernel):
    """DRAM bytes per launch recorded by ncu for `kernel`, if the kernel's
    source is unchanged since the capture (profiles/traffic.txt)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    src = {"fa_fwd_kernel": "fa_fwd.cu", "fa_bwd_main": "fa_bwd.cu"}.get(kernel)
    if src is None:
        return None
    h = hashlib.sha256()
    for f in (src, "sm103_ptx.cuh"):
        h.update(open(os.path.join(ROOT, "exact_io_aware_33_gb300", "csrc", f), "rb").read())
    digest = h.hexdigest()[:16]
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and parts[0] == kernel and parts[1] == digest:
            return float(parts[2])
    return None


def cpu_model():
    """The host CPU's model name from /proc/cpuinfo (x86: "model name"; Arm:
    implementer and part numbers), else the platform's machine name."""
    import platform
    fields = {}
    try:
        for line in open("/proc/cpuinfo"):
            if ":" in line:
                k, v = line.split(":", 1)
                fields.setdefault(k.strip().lower(), v.strip())
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    if "cpu part" in fields:
        return f"{platform.machine()} implementer {fields.get('cpu implementer', '?')} part {fields['cpu part']}"
    return platform.processor() or platform.machine()


def cpu_baseline(w, budget_s=12.0, per_config_s=2.0):
    """The float64 oracle on a bounded sample of the workload's heads, and a
    shorter bounded sample of every named workload."""
    import numpy as np  # noqa: F401
    from oracle import dense

    def run(wl, budget):
        x = si.make_inputs(wl)
        heads = [(b, h) for b in range(wl.B) for h in range(wl.H)]
        done, t0 = 0, time.perf_counter()
        for b, h in heads:
            o, lse = dense.forward_head(x["q"][b, h], x["k"][b, h], x["v"][b, h], wl.causal, wl.scale)
            if wl.backward:
                dense.backward_head(x["q"][b, h], x["k"][b, h], x["v"][b, h], o, lse, x["do"][b, h],
                                    wl.causal, wl.scale)
            done += 1
            if time.perf_counter() - t0 > budget and done >= 1:
                break
        dt = time.perf_counter() - t0
        f_fwd, f_bwd = step_flops(wl)
        return (f_fwd + f_bwd) * done / wl.heads / dt / 1e12, done, dt

    value, done, dt = run(w, budget_s)
    per_config = []
    for wl in si.WORKLOADS:
        v, n, t = run(wl, per_config_s)
        per_config.append({"workload": wl.name, "pass": "forward+backward" if wl.backward else "forward",
                           "tflops": v, "heads": f"{n} of {wl.heads}", "s": round(t, 2)})
    return {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": f"{done} of {w.heads} heads of {w.name} (dense float64 numpy "
                      f"{'forward+backward' if w.backward else 'forward'}), {dt:.1f} s",
            "os_cpu_count": os.cpu_count(), "blas_threads": blas_threads(), "cpu_model": cpu_model(),
            "per_config": per_config}


def blas_threads():
    try:
        import threadpoolctl
        import numpy  # noqa: F401
        for info in threadpoolctl.threadpool_info():
            if info.get("user_api") == "blas":
                return int(info["num_threads"])
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count()


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        barrier = lambda: dist.barrier()
    else:
        torch.cuda.set_device(0)
        barrier = lambda: None
    dev = torch.device("cuda", torch.cuda.current_device())
    w = si.workload(args.workload)
    runner = Runner(w, dev, seed_offset=rank_seed_offset(rank))
    stream = torch.cuda.Stream(dev)
    props = torch.cuda.get_device_properties(dev)
    bus = ""
    if hasattr(props, "pci_bus_id"):
        bus = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                     getattr(props, "pci_device_id", 0))
    sampler = ClockSampler(bus)
    sampler.start()
    times, wall = timed_loop(runner, args.steps, max(args.warmup, 3), barrier, stream, soak_s=1.0)
    clocks = sampler.stop()
    if clocks is not None:
        clocks["window"] = "nvidia-smi every 200 ms over warm-up, a 1 s untimed soak and the timed steps"
    mean = lambda k: sum(times[k]) / len(times[k]) if k in times else 0.0
    ms, ms_fwd, ms_bwd = max_over_ranks([mean("step"), mean("fwd"), mean("bwd_main")], dev, world)
    f_fwd, f_bwd = step_flops(w)
    value = whole_job_tflops(world, f_fwd + f_bwd, ms)
    peak, peak_sus, peak_src = measured_peaks()
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    # the dominant kernel, timed with events inside the timed region
    kernels = {"fa_bwd_main": (f_bwd, ms_bwd)} if w.backward else {"fa_fwd_kernel": (f_fwd, ms_fwd)}
    dom = max(kernels, key=lambda k: kernels[k][1])
    fl, kms = kernels[dom]
    achieved = fl / (kms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "traffic": traffic_from_profiles(dom),
                "peak_source": f"{peak_src} bf16 dense burst (MEASURED_PEAKS.json)"
                if peak_src == "measured" else "fallback 1.9 PFLOP/s"}
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded iid N(0,1) bf16 q, k, v, dO)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal, "pass": "forward+backward" if w.backward else "forward",
                   "l2": "flushed between steps (256 MiB write, outside the events)",
                   "parallelism": f"replicas x{world} (independent batches)"},
        "pct_of_peak": round(100.0 * value / (world * peak), 2),
        "kernels_ms": {k: round(v[1], 4) for k, v in kernels.items()},
        "kernels_tflops": {k: round(v[0] / (v[1] * 1e-3) / 1e12, 1) for k, v in kernels.items()},
        "kernel_events": "events around the dominant kernel in the timed region only (an event between "
                         "two kernels serialises them); the other kernels' times come from the configs leg",
        "timed_region_stats_ms": {k: {m: round(x, 4) if m != "n" else x for m, x in _stats(v).items()}
                                  for k, v in times.items()},
        "roofline": roofline,
        "gpu_launches": runner.launches_per_step * args.steps,
        "clocks": clocks,
        "wall_s": round(wall, 3),
    }
    if not args.no_extras:
        runner2 = Runner(w, dev, seed_offset=rank_seed_offset(rank))
        e_ms, h2d, d2h = e2e_loop([runner, runner2], max(3, args.steps), 2, stream)
        del runner2
        out["e2e"] = {"value": round(world * (f_fwd + f_bwd) / (e_ms * 1e-3) / 1e12, 2),
                      "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "ms_per_step": round(e_ms, 4),
                      "steps": max(3, args.steps),
                      "pipeline": "uploads, compute and downloads on three streams, two buffer sets; "
                                  "timed from the first upload to the last download"}
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        sm_mhz = (clocks or {}).get("sm_mhz") or (clocks or {}).get("sm_max_mhz") or 2070.0
        lib = runner.lib
        out["configs"] = config_legs(lib, dev, stream, runner.flush_l2, peak, sm_mhz, sms)
        if w.backward:  # the forward of this workload, from its configs record
            rec = next(r for r in out["configs"] if r["workload"] == w.name and r["pass"] == "forward")
            out["kernels_ms"]["fa_fwd_kernel"] = rec["ms_median"]
            out["kernels_tflops"]["fa_fwd_kernel"] = rec["tflops"]
        long_fwd = next(r for r in out["configs"] if r["workload"] == si.WORKLOADS[3].name)
        out["fwd_long"] = {"workload": si.WORKLOADS[3].name, "ms": long_fwd["ms_median"],
                           "tflops": long_fwd["tflops"], "frac": long_fwd["frac"]}
        out["sweep_d128"] = sweep_leg(lib, dev, stream, runner.flush_l2, peak, sm_mhz, sms)
        out["mufu_ceiling"] = {"d64": mufu_ceiling(64, sm_mhz, sms), "d128": mufu_ceiling(128, sm_mhz, sms),
                               "note": "exp2 at 32 per clock per SM (GB300, measured), one per score "
                                       "element; FLOPs per element 4d forward, 10d backward"}
        out["fwd_d256"] = d256_leg(lib, dev, stream, runner.flush_l2, peak, sm_mhz, sms)
        out["decode"] = decode_leg(dev, stream, Nk=args.decode_nk)
        out["window"] = window_leg(dev, stream, runner.flush_l2)
        out["headsize"] = headsize_leg(dev, stream, runner.flush_l2)
        out["dropout"] = dropout_leg(dev, stream, runner.flush_l2)
        if world == 1:
            out["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_only(args):
    """One extra leg alone, its JSON printed (a profiling target, not the
    bench line)."""
    import torch
    import exact_io_aware_33_gb300 as fa
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    lib = fa.load_library()
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush = flush_buf.zero_
    peak = measured_peaks()[0]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    leg = args.only
    if leg.startswith("workload:"):
        res = config_legs(lib, dev, stream, flush, peak, 2070.0, sms, names={leg.split(":", 1)[1]})
    elif leg == "configs":
        res = config_legs(lib, dev, stream, flush, peak, 2070.0, sms)
    elif leg == "sweep":
        masks = {"both": (True, False), "causal": (True,), "noncausal": (False,)}[args.sweep_causal]
        res = sweep_leg(lib, dev, stream, flush, peak, 2070.0, sms,
                        lengths=tuple(int(n) for n in args.sweep_n.split(",")), masks=masks)
    elif leg == "decode":
        res = decode_leg(dev, stream, Nk=args.decode_nk)
    elif leg == "d256":
        res = d256_leg(lib, dev, stream, flush, peak, 2070.0, sms)
    elif leg == "window":
        res = window_leg(dev, stream, flush)
    elif leg == "headsize":
        res = headsize_leg(dev, stream, flush)
    elif leg == "dropout":
        res = dropout_leg(dev, stream, flush)
    else:
        raise SystemExit(f"unknown leg {leg!r}")
    print(json.dumps({"only": leg, "result": res}), flush=True)


def run_reference(args):
    """The oracle, as it stands, on the host cores: one head per step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from oracle import dense
    w = si.workload(args.workload)
    x = si.make_inputs(w)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]

    def one(i):
        b, h = heads[i % len(heads)]
        o, lse = dense.forward_head(x["q"][b, h], x["k"][b, h], x["v"][b, h], w.causal, w.scale)
        if w.backward:
            dense.backward_head(x["q"][b, h], x["k"][b, h], x["v"][b, h], o, lse, x["do"][b, h],
                                w.causal, w.scale)

    for i in range(max(args.warmup, 3)):
        one(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(i)
    dt = (time.perf_counter() - t0) / args.steps
    f_fwd, f_bwd = step_flops(w)
    value = (f_fwd + f_bwd) / w.heads / dt / 1e12
    cores = blas_threads()
    sample = f"one head of {w.name} per step (dense float64 numpy oracle)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded iid N(0,1) bf16 q, k, v, dO upcast to float64)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal, "sample": "one (batch, head) per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
