"""Long sequences (N = 32768) through the persistent forwards, on sampled rows.

At this length one head's float64 score matrix would take 8.6 GB, so the
oracle checks rows one at a time: query row i of a causal problem is the
general-mask oracle's own sub-problem of one query over keys [0, i] (its
causal queries are the last Nq positions), and a non-causal or windowed row
is one query over every key with the window applied at its absolute
position. Rows are drawn at both ends, at 128-row tile and 256-row pair
boundaries and at random, for the one-tile (d = 64) and two-tile (d = 128)
forms. Gates as in the other forward tests: max |O - O_ref| <= 2e-2,
mean <= 2e-3, max |LSE - LSE_ref| <= 1e-3.
"""

import math

import numpy as np
import pytest
import torch as _torch_cpu

from oracle import general

torch = pytest.importorskip("torch")
fa = pytest.importorskip("exact_io_aware_33_gb300")

pytestmark = pytest.mark.gpu

N = 32768


def _rows(seed):
    rng = np.random.default_rng(seed)
    edges = [0, 1, 127, 128, 255, 256, N // 2 - 1, N // 2, N - 257, N - 256, N - 129, N - 128, N - 2, N - 1]
    return sorted(set(edges) | set(int(r) for r in rng.integers(0, N, 18)))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 4096)])
def test_long_sequence_sampled_rows(d, causal, window):
    B, H = 1, 2
    g = _torch_cpu.Generator().manual_seed(31 + d + window + (1 if causal else 0))
    q, k, v = (_torch_cpu.randn((B, H, N, d), generator=g).to(_torch_cpu.bfloat16) for _ in range(3))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fa_fwd_ex(q.cuda(), k.cuda(), v.cuda(), causal=causal, window=window, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    o = o.float().cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    errs, lse_errs = [], []
    for h in range(H):
        for i in _rows(h + d):
            if causal:  # one query at position i over keys [0, i]
                o_ref, l_ref = general.forward_head(q[0, h, i:i + 1], k[0, h, :i + 1], v[0, h, :i + 1],
                                                    True, scale, window)
            else:  # one query over every key
                o_ref, l_ref = general.forward_head(q[0, h, i:i + 1], k[0, h], v[0, h], False, scale, window)
            errs.append(np.abs(o[0, h, i] - o_ref[0]))
            lse_errs.append(abs(lse[0, h, i] - l_ref[0]))
    err = np.stack(errs)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
    assert max(lse_errs) <= 1e-3
