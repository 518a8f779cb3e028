"""Head size d = d_v = 256 in the forward forms, on the GPU against the
float64 oracle.

The pages count the forward's work as O(N^2 (d + d_v)) ("Flash Attention:
IO-Aware Exact Attention", section "Storage, arithmetic and IO are separate
quantities"); d = 256 runs one 128-row query tile per CTA, whose S (128
columns) and O accumulator (256 columns) fill the tensor memory. Forward
gate as everywhere: max |O - O_ref| <= 2e-2, mean <= 2e-3, max |LSE -
LSE_ref| <= 1e-3, over every element. The backward does not take d = 256 and
must say so (FA_ERR_UNSUPPORTED) without launching anything.
"""

import ctypes
import math

import numpy as np
import pytest

import synthetic_inputs as si
from oracle import dense, general

torch = pytest.importorskip("torch")
fa = pytest.importorskip("exact_io_aware_33_gb300")

pytestmark = pytest.mark.gpu

D = 256


def _check_fwd(o, lse, o_ref, lse_ref):
    err = np.abs(o.float().cpu().double().numpy() - o_ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
    assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= 1e-3


def _inputs(B, H, Nq, Nk, seed, k_mult=1.0):
    q = si.make_small(B, H, Nq, D, seed=seed, with_grad=False)["q"]
    kv = si.make_small(B, H, Nk, D, seed=seed + 1, k_mult=k_mult, with_grad=False)
    return q, kv["k"], kv["v"]


@pytest.mark.parametrize("B,H,N,causal", [
    (1, 1, 256, False),
    (1, 2, 300, True),     # ragged tail
    (2, 1, 1000, False),   # several key tiles, ragged
    (1, 1, 1, True),       # a lone row
    (1, 3, 640, True),     # causal diagonal tiles
])
def test_forward_d256(B, H, N, causal):
    x = si.make_small(B, H, N, D, seed=5000 + N + B, with_grad=False)
    scale = 1.0 / math.sqrt(D)
    o, lse = fa.fa_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    _check_fwd(o, lse, *dense.forward(x["q"], x["k"], x["v"], causal, scale))


def test_forward_d256_large_scores_move_the_maximum():
    # keys x8: row maxima jump across key tiles, exercising the rescale of the 256-column O.
    # With scores this peaked each output row is nearly one value row; V is halved (exactly,
    # in bf16) so that |O| < 4 and the bf16 rounding of O itself (half a unit in the last
    # place, 2^-7 below 4 but 2^-6 from 4 to 8) leaves the gate room for the kernel's error.
    q, k, v = _inputs(1, 2, 700, 700, seed=77, k_mult=8.0)
    v = (v.float() * 0.5).to(v.dtype)
    scale = 1.0 / math.sqrt(D)
    for causal in (False, True):
        o, lse = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
        torch.cuda.synchronize()
        _check_fwd(o, lse, *dense.forward(q, k, v, causal, scale))


@pytest.mark.parametrize("Nq,Nk,causal,window", [(300, 1000, True, 0), (256, 333, False, 0),
                                                 (700, 700, True, 200), (5, 4096, True, 0)])
def test_forward_ex_d256(Nq, Nk, causal, window):
    q, k, v = _inputs(1, 2, Nq, Nk, seed=Nq + Nk + window)
    scale = 1.0 / math.sqrt(D)
    o, lse = fa.fa_fwd_ex(q.cuda(), k.cuda(), v.cuda(), causal=causal, window=window, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    assert tuple(o.shape) == (1, 2, Nq, D)
    _check_fwd(o, lse, *general.forward(q, k, v, causal, scale, window))


@pytest.mark.parametrize("Nq,splits", [(1, 0), (3, 5), (130, 4)])
def test_decode_splitkv_d256(Nq, splits):
    q, k, v = _inputs(2, 4, Nq, 3000, seed=900 + Nq)
    scale = 1.0 / math.sqrt(D)
    o, lse = fa.fa_decode_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale,
                                  n_splits=splits)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    _check_fwd(o, lse, *general.forward(q, k, v, True, scale))


def test_forward_d256_bench_shape_every_head():
    # the bench's d = 256 point (causal, N=4096) on 4 heads, every head compared
    B, H, N = 1, 4, 4096
    x = si.make_small(B, H, N, D, seed=256, with_grad=False)
    scale = 1.0 / math.sqrt(D)
    o, lse = fa.fa_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    _check_fwd(o, lse, *dense.forward(x["q"], x["k"], x["v"], True, scale))


def test_backward_refuses_d256_and_mixed_sizes():
    lib = fa.load_library()
    t = torch.zeros(1 << 16, dtype=torch.bfloat16, device="cuda")  # never read: refused first
    p = ctypes.c_void_p(t.data_ptr())
    z = ctypes.c_void_p(0)
    assert lib.fa_bwd(p, p, p, p, p, p, p, p, p, 1, 1, 64, D, 1, 0.0625) == fa.FA_ERR_UNSUPPORTED
    ws = lib.fa_bwd_workspace_bytes(1, 1, 64, D)
    assert lib.fa_bwd_stream(p, p, p, p, p, p, p, p, p, 1, 1, 64, D, 1, 0.0625, p, ws, z) == \
        fa.FA_ERR_UNSUPPORTED
    assert lib.fa_bwd_ex(p, p, p, p, p, p, p, p, p, 1, 1, 64, D, D, 1, 0, 0.0625, p, ws, z) == \
        fa.FA_ERR_UNSUPPORTED
    assert lib.fa_bwd_dropout(p, p, p, p, p, p, p, p, p, 1, 1, 64, D, 1, 0.0625, 0.1, 1, 0, p, ws,
                              z) == fa.FA_ERR_UNSUPPORTED
    # d = 256 pairs only with d_v = 256
    assert lib.fa_fwd_ex(p, p, p, p, p, 1, 1, 8, 8, D, 64, 0, 0, 0.1, z) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_fwd_ex(p, p, p, p, p, 1, 1, 8, 8, 128, D, 0, 0, 0.1, z) == fa.FA_ERR_UNSUPPORTED
    # dropout is not offered at d = 256
    assert lib.fa_fwd_dropout(p, p, p, p, p, 1, 1, 64, D, 1, 0.0625, 0.1, 1, 0, z) == \
        fa.FA_ERR_UNSUPPORTED
