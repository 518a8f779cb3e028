"""Extended forward on the GPU against the float64 general-mask oracle.

fa_fwd_ex: Nq queries over Nk keys (causal queries are the last Nq
positions, as in a decode step over a key/value cache) and sliding windows.
fa_decode_splitkv: the same result computed as partial states over split key
ranges and merged with the rule of "FlashAttention -- the same attention,
made memory-aware", section 03. Tolerances are the forward's: max |O - O_ref|
<= 2e-2, mean <= 2e-3, max |LSE - LSE_ref| <= 1e-3.
"""

import math

import numpy as np
import pytest

import synthetic_inputs as si
from oracle import general

torch = pytest.importorskip("torch")
fa = pytest.importorskip("exact_io_aware_33_gb300")

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


def _inputs(B, H, Nq, Nk, d, seed):
    q = si.make_small(B, H, Nq, d, seed=seed, with_grad=False)["q"]
    kv = si.make_small(B, H, Nk, d, seed=seed + 1, with_grad=False)
    return q, kv["k"], kv["v"]


def _check(o, lse, q, k, v, causal, window, scale, heads=None):
    o_ref, lse_ref = general.forward(q, k, v, causal, scale, window, heads=heads)
    o = o.float().cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    if heads is not None:
        o = np.stack([o[b, h] for b, h in heads])
        lse = np.stack([lse[b, h] for b, h in heads])
        o_ref = np.stack([o_ref[b, h] for b, h in heads])
        lse_ref = np.stack([lse_ref[b, h] for b, h in heads])
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())
    assert np.abs(lse - lse_ref).max() <= LSE_MAX


CASES = [
    # B, H, Nq, Nk, d, causal, window
    (1, 2, 1, 1000, 64, True, 0),       # one decode query over a ragged cache
    (2, 2, 7, 2048, 128, True, 0),      # a few decode queries
    (1, 2, 300, 1000, 64, True, 0),     # chunked prefill: several query tiles, offset diagonal
    (1, 1, 256, 333, 128, False, 0),    # cross attention, more keys than queries
    (1, 2, 500, 200, 64, False, 0),     # cross attention, more queries than keys
    (1, 2, 640, 640, 64, True, 1),      # window of one key: O = V at the own position
    (1, 2, 700, 700, 128, True, 100),   # window inside a tile
    (2, 1, 1000, 1000, 64, True, 256),  # window of two tiles, ragged N
    (1, 2, 512, 1536, 128, True, 300),  # window with an offset
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,window", CASES)
def test_fwd_ex_matches_oracle(B, H, Nq, Nk, d, causal, window):
    q, k, v = _inputs(B, H, Nq, Nk, d, seed=Nq * 7 + Nk + d + window)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fa_fwd_ex(q.cuda(), k.cuda(), v.cuda(), causal=causal, window=window, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    _check(o, lse, q, k, v, causal, window, scale)


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,window,splits", [
    (2, 4, 1, 4096, 64, True, 0, 0),
    (1, 8, 4, 3000, 128, True, 0, 5),
    (1, 2, 16, 1024, 64, False, 0, 3),
    (1, 2, 130, 2000, 64, True, 0, 4),    # two query tiles per CTA
    (1, 2, 8, 4096, 128, True, 700, 6),   # window: most splits see no key for most rows
    (1, 1, 3, 300, 64, True, 0, 64),      # more splits asked than key tiles
])
def test_decode_splitkv_matches_oracle(B, H, Nq, Nk, d, causal, window, splits):
    q, k, v = _inputs(B, H, Nq, Nk, d, seed=Nk + Nq + splits)
    scale = 1.0 / math.sqrt(d)
    used = fa.fa_decode_num_splits(B, H, Nq, Nk, splits)
    assert 1 <= used <= -(-Nk // 128)
    o, lse = fa.fa_decode_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=causal, window=window,
                                  scale=scale, n_splits=splits)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    _check(o, lse, q, k, v, causal, window, scale)
    # the split result agrees with the one-pass extended forward
    o1, lse1 = fa.fa_fwd_ex(q.cuda(), k.cuda(), v.cuda(), causal=causal, window=window, scale=scale)
    torch.cuda.synchronize()
    assert (o.float() - o1.float()).abs().max().item() <= 2e-2
    assert (lse - lse1).abs().max().item() <= 1e-3


@pytest.mark.parametrize("causal,window", [(True, 0), (True, 200), (False, 0)])
def test_fwd_ex_many_ctas_per_sm(causal, window):
    # d = 64 runs one query tile per CTA, two CTAs per SM: 4 x 32 heads x 3
    # query tiles = 384 CTAs of different key ranges (offset diagonal, window,
    # ragged tails) share the SMs; every head compared.
    B, H, Nq, Nk, d = 4, 32, 333, 800, 64
    q, k, v = _inputs(B, H, Nq, Nk, d, seed=901 + window + int(causal))
    scale = 0.125
    o, lse = fa.fa_fwd_ex(q.cuda(), k.cuda(), v.cuda(), causal=causal, window=window, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    _check(o, lse, q, k, v, causal, window, scale)


def test_fwd_ex_square_equals_fa_fwd():
    q, k, v = _inputs(2, 3, 777, 777, 64, seed=5)
    a = fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    b = fa.fa_fwd_ex(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_decode_long_cache_every_head():
    # B=8 H=32 Nq=1 Nk=32768 d=128, causal: the decode workload at full size,
    # every one of the 256 heads compared.
    B, H, Nq, Nk, d = 8, 32, 1, 32768, 128
    q, k, v = _inputs(B, H, Nq, Nk, d, seed=31)
    o, lse = fa.fa_decode_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    _check(o, lse, q, k, v, True, 0, 1.0 / math.sqrt(d))


def test_invalid_extended_arguments_are_refused():
    lib = fa.load_library()
    t = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    p = __import__("ctypes").c_void_p(t.data_ptr())
    z = __import__("ctypes").c_void_p(0)
    # window without causal, negative window, causal with more queries than keys
    assert lib.fa_fwd_ex(p, p, p, p, p, 1, 1, 8, 8, 64, 64, 0, 4, 0.1, z) == fa.FA_ERR_INVALID
    assert lib.fa_fwd_ex(p, p, p, p, p, 1, 1, 8, 8, 64, 64, 1, -1, 0.1, z) == fa.FA_ERR_INVALID
    assert lib.fa_fwd_ex(p, p, p, p, p, 1, 1, 9, 8, 64, 64, 1, 0, 0.1, z) == fa.FA_ERR_INVALID
    # no keys for live queries
    assert lib.fa_fwd_ex(p, p, p, p, p, 1, 1, 8, 0, 64, 64, 0, 0, 0.1, z) == fa.FA_ERR_INVALID
    # empty query set: nothing to do
    assert lib.fa_fwd_ex(z, z, z, z, z, 1, 1, 0, 8, 64, 64, 0, 0, 0.1, z) == fa.FA_OK
    # split form without a large enough workspace
    assert lib.fa_decode_splitkv(p, p, p, p, p, 1, 1, 1, 4096, 64, 64, 1, 0, 0.1, 4, p, 16, z) == \
        fa.FA_ERR_WORKSPACE
