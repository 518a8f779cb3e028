"""Backward with causal sliding windows on the GPU against the float64
general-mask oracle (window W: a query at position i sees keys i-W < j <= i;
"Flash Attention: IO-Aware Exact Attention", section "What changes in
FlashAttention-2", sliding-window attention). Gate: per tensor,
||dX - dX_ref||_inf / ||dX_ref||_inf <= 5e-2.
"""

import math

import numpy as np
import pytest

import synthetic_inputs as si
from oracle import general

torch = pytest.importorskip("torch")
fa = pytest.importorskip("exact_io_aware_33_gb300")

pytestmark = pytest.mark.gpu

REL = 5e-2


@pytest.mark.parametrize("B,H,N,d,window", [
    (1, 2, 384, 64, 1),
    (1, 2, 700, 64, 100),
    (2, 1, 1000, 64, 256),
    (1, 2, 640, 128, 128),
    (1, 1, 900, 128, 300),
    (1, 2, 512, 64, 2000),   # wider than the sequence: plain causal
])
def test_windowed_backward_matches_oracle(B, H, N, d, window):
    x = si.make_small(B, H, N, d, seed=N + window + d, with_grad=True)
    g = {k: t.cuda() for k, t in x.items()}
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fa_fwd_ex(g["q"], g["k"], g["v"], causal=True, window=window, scale=scale)
    dq, dk, dv = fa.fa_bwd_ex(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True, window=window,
                              scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    o_ref, lse_ref = general.forward(x["q"], x["k"], x["v"], True, scale, window)
    ref = general.backward(x["q"], x["k"], x["v"], o_ref, lse_ref, x["do"], True, scale, window)
    dv_scale = np.abs(ref[2]).max()
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        gg = got.float().cpu().double().numpy()
        # A window of one key makes P the identity and dS = P * (dP - D)
        # vanish, so dQ and dK are exactly zero: gate them against dV's scale.
        denom = np.abs(r).max() if np.abs(r).max() > 1e-9 * dv_scale else dv_scale
        rel = np.abs(gg - r).max() / denom
        assert rel <= REL, (name, rel)


def test_windowed_backward_many_items_per_cta():
    # 4 x 24 heads x 5 key blocks = 480 items, about three per CTA of the
    # persistent d = 64 kernel, each stopping at the last query block its
    # window reaches; ragged last block; compared on every head.
    B, H, N, d, window = 4, 24, 600, 64, 150
    x = si.make_small(B, H, N, d, seed=91, with_grad=True)
    g = {k: t.cuda() for k, t in x.items()}
    scale = 0.125
    o, lse = fa.fa_fwd_ex(g["q"], g["k"], g["v"], causal=True, window=window, scale=scale)
    dq, dk, dv = fa.fa_bwd_ex(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True, window=window,
                              scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    o_ref, lse_ref = general.forward(x["q"], x["k"], x["v"], True, scale, window)
    ref = general.backward(x["q"], x["k"], x["v"], o_ref, lse_ref, x["do"], True, scale, window)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        rel = np.abs(got.float().cpu().double().numpy() - r).max() / np.abs(r).max()
        assert rel <= REL, (name, rel)


def test_wide_window_backward_equals_causal_backward():
    x = si.make_small(1, 2, 600, 64, seed=3, with_grad=True)
    g = {k: t.cuda() for k, t in x.items()}
    o, lse = fa.fa_fwd(g["q"], g["k"], g["v"], causal=True)
    a = fa.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True)
    b = fa.fa_bwd_ex(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True, window=600)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert (a[0].float() - b[0].float()).abs().max().item() <= 1e-2
