"""Seeded random sweep of small problems on the GPU against the float64
general-mask oracle ("Flash Attention: IO-Aware Exact Attention", sections
"Online softmax makes tiling exact" and "What changes in FlashAttention-2"):
head sizes d, d_v in {64, 128}, causal or not, causal windows, Nq <= Nk with
the queries at the end of the keys (decode-style offsets), ragged lengths.
Forward and (for Nq = Nk) backward are compared element by element on every
head with the gates of the dedicated parity tests.
"""
import numpy as np
import pytest

import synthetic_inputs as si
from oracle import general

torch = pytest.importorskip("torch")
fa = pytest.importorskip("exact_io_aware_33_gb300")

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX, GRAD_REL = 2e-2, 2e-3, 1e-3, 5e-2


def _configs(n, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        d = int(rng.choice([64, 128]))
        dv = int(rng.choice([64, 128]))
        nk = int(rng.integers(1, 700))
        square = bool(rng.integers(0, 2))
        nq = nk if square else int(rng.integers(1, nk + 1))
        causal = bool(rng.integers(0, 3) > 0)
        window = int(rng.choice([0, 0, 1, 37, 128, 300])) if causal else 0
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        out.append((B, H, nq, nk, d, dv, causal, window))
    return out


CONFIGS = _configs(16)


@pytest.mark.parametrize("B,H,Nq,Nk,d,dv,causal,window", CONFIGS)
def test_random_config_matches_oracle(B, H, Nq, Nk, d, dv, causal, window):
    seed = B * 1000003 + H * 10007 + Nq * 101 + Nk + d + dv + window
    q = si.make_small(B, H, Nq, d, seed=seed)["q"]
    kv = si.make_small(B, H, Nk, max(d, dv), seed=seed + 1)
    k = kv["k"][..., :d].contiguous()
    v = kv["v"][..., :dv].contiguous()
    scale = 1.0 / np.sqrt(d)
    g = [t.cuda() for t in (q, k, v)]
    o, lse = fa.fa_fwd_ex(*g, causal=causal, window=window, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    o_ref, lse_ref = general.forward(q, k, v, causal, scale, window)
    err = np.abs(o.float().cpu().double().numpy() - o_ref)
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())
    lse_g = lse.cpu().double().numpy()
    finite = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_g), finite)
    assert np.abs(lse_g[finite] - lse_ref[finite]).max(initial=0.0) <= LSE_MAX
    if Nq != Nk:
        return
    do = si.make_small(B, H, Nq, dv, seed=seed + 2)["q"]
    dq, dk, dv_ = fa.fa_bwd_ex(*g, o, lse, do.cuda(), causal=causal, window=window, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    ref = general.backward(q, k, v, o_ref, lse_ref, do, causal, scale, window)
    scale_ref = max(np.abs(r).max() for r in ref)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv_), ref):
        gg = got.float().cpu().double().numpy()
        # a window of one key makes dS vanish (dQ = dK = 0): gate against the largest gradient
        denom = np.abs(r).max() if np.abs(r).max() > 1e-9 * scale_ref else scale_ref
        assert np.abs(gg - r).max() / denom <= GRAD_REL, (name, np.abs(gg - r).max() / denom)
