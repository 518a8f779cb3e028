"""Head sizes: d (queries, keys) and d_v (values, output) each 64 or 128, on
the GPU against the float64 general-mask oracle. The pages count the
forward's work as O(N^2 (d + d_v)) ("Flash Attention: IO-Aware Exact
Attention", section "Storage, arithmetic and IO are separate quantities"),
with d_v = d as the square special case. Forward gate: max |O - O_ref| <=
2e-2, mean <= 2e-3, max |LSE - LSE_ref| <= 1e-3; backward gate:
||dX - dX_ref||_inf / ||dX_ref||_inf <= 5e-2 per tensor.
"""

import math

import numpy as np
import pytest
import torch as _torch_cpu

from oracle import general

torch = pytest.importorskip("torch")
fa = pytest.importorskip("exact_io_aware_33_gb300")

pytestmark = pytest.mark.gpu


def _draw(shape, g):
    return _torch_cpu.randn(shape, generator=g, dtype=_torch_cpu.float32).to(_torch_cpu.bfloat16)


def _inputs(B, H, Nq, Nk, d, dv, seed, grad=False):
    g = _torch_cpu.Generator().manual_seed(seed)
    x = {"q": _draw((B, H, Nq, d), g), "k": _draw((B, H, Nk, d), g), "v": _draw((B, H, Nk, dv), g)}
    if grad:
        x["do"] = _draw((B, H, Nq, dv), g)
    return x


def _check_fwd(o, lse, o_ref, lse_ref):
    err = np.abs(o.float().cpu().double().numpy() - o_ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
    assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= 1e-3


@pytest.mark.parametrize("d,dv", [(128, 64), (64, 128)])
@pytest.mark.parametrize("Nq,Nk,causal,window", [(640, 640, True, 0), (300, 1000, True, 0),
                                                 (256, 333, False, 0), (700, 700, True, 200)])
def test_forward_head_sizes(d, dv, Nq, Nk, causal, window):
    x = _inputs(1, 2, Nq, Nk, d, dv, seed=d * 3 + dv + Nq + Nk + window)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fa_fwd_ex(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=causal, window=window,
                          scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    assert tuple(o.shape) == (1, 2, Nq, dv)
    _check_fwd(o, lse, *general.forward(x["q"], x["k"], x["v"], causal, scale, window))


@pytest.mark.parametrize("d,dv", [(128, 64), (64, 128)])
def test_decode_head_sizes(d, dv):
    x = _inputs(2, 4, 3, 3000, d, dv, seed=d + dv)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fa_decode_splitkv(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=True,
                                  scale=scale, n_splits=5)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    _check_fwd(o, lse, *general.forward(x["q"], x["k"], x["v"], True, scale))


@pytest.mark.parametrize("d,dv", [(128, 64), (64, 128), (128, 128), (64, 64)])
@pytest.mark.parametrize("N,causal,window", [(640, True, 0), (1000, False, 0), (900, True, 300)])
def test_backward_head_sizes(d, dv, N, causal, window):
    x = _inputs(1, 2, N, N, d, dv, seed=7 * d + dv + N + window, grad=True)
    g = {k: t.cuda() for k, t in x.items()}
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fa_fwd_ex(g["q"], g["k"], g["v"], causal=causal, window=window, scale=scale)
    dq, dk, dvv = fa.fa_bwd_ex(g["q"], g["k"], g["v"], o, lse, g["do"], causal=causal,
                               window=window, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    o_ref, lse_ref = general.forward(x["q"], x["k"], x["v"], causal, scale, window)
    ref = general.backward(x["q"], x["k"], x["v"], o_ref, lse_ref, x["do"], causal, scale, window)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dvv), ref):
        gg = got.float().cpu().double().numpy()
        rel = np.abs(gg - r).max() / np.abs(r).max()
        assert rel <= 5e-2, (name, rel)
