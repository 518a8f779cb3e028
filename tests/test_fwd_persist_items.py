"""The persistent forwards over many items per CTA, against the float64
general-mask oracle.

A persistent CTA keeps its barriers, K/V ring and tensor memory across the
query tiles (or pairs of query tiles) it is dealt, so every barrier phase runs
on counts over all of them. These cases give each CTA several items, some of
whose second query tile lies past the last row (an odd number of 128-row
tiles) and whose last tile is ragged, for each head-size pair, causal and not,
with and without a window: a phase that a skipped tile or a short item put
out of step would show as wrong rows, or as a bounded wait running out.
Gates as in the other forward tests: max |O - O_ref| <= 2e-2, mean <= 2e-3,
max |LSE - LSE_ref| <= 1e-3, every head.
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


@pytest.mark.parametrize("d,dv", [(128, 128), (128, 64), (64, 128), (64, 64)])
@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 200)])
def test_many_items_per_cta(d, dv, causal, window):
    # B * H = 160 heads of N = 300: three query tiles per head (the third
    # ragged), so 320 pairs or 480 tiles over one or two CTAs per SM
    B, H, N = 4, 40, 300
    g = _torch_cpu.Generator().manual_seed(d + 7 * dv + (3 if causal else 0) + window)
    q, k, v = _draw((B, H, N, d), g), _draw((B, H, N, d), g), _draw((B, H, N, dv), g)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fa_fwd_ex(q.cuda(), k.cuda(), v.cuda(), causal=causal, window=window, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    o_ref, lse_ref = general.forward(q, k, v, causal, scale, window)
    err = np.abs(o.float().cpu().double().numpy() - o_ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
    assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= 1e-3
