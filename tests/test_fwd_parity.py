"""Forward pass on the GPU against the float64 CPU oracle.

Tolerances (bf16 inputs, fp32 accumulation): max |O - O_ref| <= 2e-2,
mean |O - O_ref| <= 2e-3, max |LSE - LSE_ref| <= 1e-3, over every element
compared. Small problems and the five named workloads at full size are all
compared element by element on every head; properties that hold at any size
(finite outputs, outputs inside the convex hull of the values) are checked
on top.
"""

import math

import numpy as np
import pytest

import synthetic_inputs as si
from oracle import dense

torch = pytest.importorskip("torch")
fa = pytest.importorskip("exact_io_aware_33_gb300")

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


def _gpu(x):
    return {k: t.cuda() for k, t in x.items()}


def _compare(o, lse, o_ref, lse_ref, heads=None):
    o = o.float().cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    if heads is not None:
        o = np.stack([o[b, h] for b, h in heads])
        lse = np.stack([lse[b, h] for b, h in heads])
        o_ref = np.stack([o_ref[b, h] for b, h in heads])
        lse_ref = np.stack([lse_ref[b, h] for b, h in heads])
    err = np.abs(o - o_ref)
    lerr = np.abs(lse - lse_ref)
    assert err.max() <= O_MAX, f"max |O - O_ref| = {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"mean |O - O_ref| = {err.mean():.3e}"
    assert lerr.max() <= LSE_MAX, f"max |LSE - LSE_ref| = {lerr.max():.3e}"
    return err.max(), err.mean(), lerr.max()


def _run(x, causal, scale):
    g = _gpu(x)
    o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    return o, lse


SMALL = [
    # B, H, N, d, causal  -- several tiles, ragged tails, a lone row, both head sizes
    (1, 1, 256, 64, False),
    (1, 2, 128, 64, True),
    (2, 2, 129, 64, True),
    (1, 1, 1, 64, False),
    (1, 1, 1, 128, True),
    (1, 3, 300, 128, False),
    (2, 1, 513, 64, True),
    (1, 2, 1000, 128, True),
    (1, 1, 127, 128, False),
    (3, 1, 255, 64, False),
    (1, 1, 384, 128, True),
    (1, 2, 640, 64, False),
]


@pytest.mark.parametrize("B,H,N,d,causal", SMALL)
def test_small_against_oracle(B, H, N, d, causal):
    x = si.make_small(B, H, N, d, seed=1000 + N + d + B, with_grad=False)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(x, causal, scale)
    o_ref, lse_ref = dense.forward(x["q"], x["k"], x["v"], causal, scale)
    _compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_workload_full_size(idx):
    w = si.WORKLOADS[idx]
    x = si.make_inputs(w, with_grad=False)
    o, lse = _run(x, w.causal, w.scale)
    # every head, element by element
    o_ref, lse_ref = dense.forward(x["q"], x["k"], x["v"], w.causal, w.scale)
    _compare(o, lse, o_ref, lse_ref)
    # finite, and each output row inside the values' range
    of = o.float()
    assert torch.isfinite(of).all() and torch.isfinite(lse).all()
    vf = x["v"].float().cuda()
    vmax = vf.amax(dim=2, keepdim=True)
    vmin = vf.amin(dim=2, keepdim=True)
    slack = 1e-2 * (vmax - vmin) + 1e-2
    assert bool((of <= vmax + slack).all()) and bool((of >= vmin - slack).all())


@pytest.mark.parametrize("d", [64, 128])
def test_scale_zero_is_uniform_average(d):
    x = si.make_small(1, 2, 300, d, seed=5, with_grad=False)
    for causal in (False, True):
        o, lse = _run(x, causal, 0.0)
        o_ref, lse_ref = dense.forward(x["q"], x["k"], x["v"], causal, 0.0)
        _compare(o, lse, o_ref, lse_ref)


def test_large_scores_move_the_maximum():
    # keys scaled x8: row maxima jump across tiles, exercising the rescale
    x = si.make_small(1, 2, 700, 128, seed=9, k_mult=8.0, with_grad=False)
    for causal in (False, True):
        o, lse = _run(x, causal, 1.0 / math.sqrt(128))
        o_ref, lse_ref = dense.forward(x["q"], x["k"], x["v"], causal, 1.0 / math.sqrt(128))
        _compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("d", [64, 128])
def test_deterministic(d):
    x = si.make_small(2, 3, 777, d, seed=11, with_grad=False)
    o1, l1 = _run(x, True, 0.125)
    o2, l2 = _run(x, True, 0.125)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d", [64, 128])
def test_rows_beyond_n_untouched(d):
    # outputs live in a larger buffer; the bytes after the problem stay as set
    B, H, N = 1, 1, 200
    x = si.make_small(B, H, N, d, seed=13, with_grad=False)
    g = _gpu(x)
    big = torch.full((B * H * N * d + 4096,), float("nan"), dtype=torch.bfloat16, device="cuda")
    lbig = torch.full((B * H * N + 1024,), float("nan"), dtype=torch.float32, device="cuda")
    o = big[: B * H * N * d].view(B, H, N, d)
    lse = lbig[: B * H * N].view(B, H, N)
    fa.fa_fwd(g["q"], g["k"], g["v"], causal=True, scale=0.125, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.isnan(big[B * H * N * d:]).all()
    assert torch.isnan(lbig[B * H * N:]).all()
    assert torch.isfinite(o.float()).all()


def test_empty_and_invalid():
    z = torch.zeros(1, 1, 0, 64, dtype=torch.bfloat16, device="cuda")
    o, lse = fa.fa_fwd(z, z, z)
    assert o.shape == (1, 1, 0, 64)
    x = torch.zeros(1, 1, 8, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd(x, x, x)
    assert e.value.code == fa.FA_ERR_UNSUPPORTED
    y = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd(y, y, y, scale=float("nan"))
    assert e.value.code == fa.FA_ERR_INVALID


def test_no_quadratic_memory():
    # the long causal workload must not allocate anything that grows with N^2
    w = si.WORKLOADS[3]
    x = _gpu(si.make_inputs(w, with_grad=False))
    o = torch.empty_like(x["q"])
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    torch.cuda.reset_peak_memory_stats()
    before = torch.cuda.memory_allocated()
    fa.fa_fwd(x["q"], x["k"], x["v"], causal=True, scale=w.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.max_memory_allocated() == before
    s_bytes = 4 * w.B * w.H * w.N * w.N
    assert free0 - free1 < s_bytes // 64
