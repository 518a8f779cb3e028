"""Pins of the general-mask oracle and of the partial-state merge (no GPU).

``oracle.general`` extends the dense definition to Nq queries over Nk keys
(causal queries are the last Nq positions: a decode step over a key/value
cache) and to sliding windows; ``oracle.merge`` is the rule of
"FlashAttention -- the same attention, made memory-aware", section 03, for
combining partial softmax states. Each test below fixes them by something
other than their own formulas.
"""

import math

import numpy as np
import pytest

from oracle import dense, finite_diff, general, merge

RNG = np.random.default_rng(20260)


def _qkv(nq, nk, d, dv=None, seed=0):
    g = np.random.default_rng(seed)
    dv = dv or d
    return g.standard_normal((nq, d)), g.standard_normal((nk, d)), g.standard_normal((nk, dv))


def _brute(q, k, v, causal, scale, window):
    """Per row: softmax over an explicit slice of the visible keys."""
    nq, nk = q.shape[0], k.shape[0]
    off = nk - nq
    o = np.zeros((nq, v.shape[1]))
    lse = np.full(nq, -np.inf)
    for i in range(nq):
        hi = min(nk, i + off + 1) if causal else nk
        lo = max(0, i + off - window + 1) if window else 0
        if hi <= lo:
            continue
        s = np.array([scale * float(np.dot(q[i], k[j])) for j in range(lo, hi)])
        m = s.max()
        e = np.exp(s - m)
        o[i] = (e[:, None] * v[lo:hi]).sum(axis=0) / e.sum()
        lse[i] = m + math.log(e.sum())
    return o, lse


@pytest.mark.parametrize("nq,nk,causal,window", [
    (5, 5, False, 0), (5, 5, True, 0), (3, 9, True, 0), (1, 7, True, 0), (4, 10, False, 0),
    (6, 6, True, 2), (6, 6, True, 1), (3, 11, True, 4), (8, 8, True, 3), (2, 9, True, 20),
])
def test_general_matches_brute_force_slices(nq, nk, causal, window):
    q, k, v = _qkv(nq, nk, 3, seed=nq * 100 + nk)
    o, lse = general.forward_head(q, k, v, causal, 0.7, window)
    ob, lb = _brute(q, k, v, causal, 0.7, window)
    np.testing.assert_allclose(o, ob, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lb, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_general_equals_dense_when_square_and_unwindowed(causal):
    q, k, v = _qkv(9, 9, 4, seed=3)
    o, lse = general.forward_head(q, k, v, causal, 0.5)
    od, ld = dense.forward_head(q, k, v, causal, 0.5)
    np.testing.assert_allclose(o, od, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, ld, rtol=1e-13, atol=1e-13)


def test_window_one_selects_the_own_position():
    q, k, v = _qkv(4, 7, 3, seed=5)
    o, lse = general.forward_head(q, k, v, True, 0.3, window=1)
    off = 3
    for i in range(4):
        np.testing.assert_allclose(o[i], v[i + off], rtol=0, atol=1e-15)
        assert abs(lse[i] - 0.3 * float(q[i] @ k[i + off])) < 1e-14


def test_wide_window_equals_plain_causal_and_decode_row_sees_all_keys():
    q, k, v = _qkv(5, 12, 4, seed=6)
    a = general.forward_head(q, k, v, True, 0.4, window=12)
    b = general.forward_head(q, k, v, True, 0.4, window=0)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-14, atol=1e-14)
    q1 = q[-1:]
    c = general.forward_head(q1, k, v, True, 0.4)
    d = general.forward_head(q1, k, v, False, 0.4)
    np.testing.assert_allclose(c[0], d[0], rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("nq,nk,window", [(4, 4, 0), (4, 4, 2), (3, 6, 0), (5, 5, 3)])
def test_general_backward_matches_finite_differences(nq, nk, window):
    q, k, v = _qkv(nq, nk, 3, seed=nq + nk + window)
    do = np.random.default_rng(9).standard_normal((nq, 3))
    o, lse = general.forward_head(q, k, v, True, 0.6, window)
    g = general.backward_head(q, k, v, o, lse, do, True, 0.6, window)
    n = finite_diff.gradients_general(q, k, v, do, True, 0.6, window)
    for a, b in zip(g, n):
        np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-7)


def test_general_backward_equals_dense_when_square():
    q, k, v = _qkv(7, 7, 4, seed=11)
    do = np.random.default_rng(12).standard_normal((7, 4))
    o, lse = dense.forward_head(q, k, v, True, 0.5)
    for a, b in zip(general.backward_head(q, k, v, o, lse, do, True, 0.5),
                    dense.backward_head(q, k, v, o, lse, do, True, 0.5)):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("nq,nk,causal,window,bounds", [
    (3, 20, True, 0, [0, 7, 13, 20]),
    (1, 33, True, 0, [0, 1, 2, 16, 33]),
    (6, 6, True, 3, [0, 2, 3, 6]),
    (4, 9, False, 0, [0, 9]),
    (5, 17, True, 6, [0, 4, 8, 12, 17]),     # some parts see no key for some rows
])
def test_merged_parts_equal_the_whole(nq, nk, causal, window, bounds):
    q, k, v = _qkv(nq, nk, 4, seed=nk)
    parts = [general.forward_head(q, k, v, causal, 0.45, window, key_range=(a, b))
             for a, b in zip(bounds[:-1], bounds[1:])]
    o, lse = merge.merge(parts)
    ow, lw = general.forward_head(q, k, v, causal, 0.45, window)
    np.testing.assert_allclose(o, ow, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lw, rtol=1e-12, atol=1e-12)
    # any order of merging gives the same result
    o2, l2 = merge.merge(parts[::-1])
    np.testing.assert_allclose(o2, ow, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l2, lw, rtol=1e-12, atol=1e-12)


def test_merge_reproduces_the_pages_running_sum():
    # scores [1, 3] then [2, 5], each reduced on its own to (m, l)
    m1, l1 = 3.0, math.exp(1 - 3) + 1.0
    m2, l2 = 5.0, math.exp(2 - 5) + 1.0
    o = np.zeros((1, 1))
    m, l, _ = merge.merge_two(np.array([m1]), np.array([l1]), o, np.array([m2]), np.array([l2]), o)
    assert m[0] == 5.0
    assert round(l[0], 3) == 1.203
    # the same through the saved-statistic form
    _, lse = merge.merge([(o, np.array([m1 + math.log(l1)])), (o, np.array([m2 + math.log(l2)]))])
    assert round(math.exp(lse[0] - 5.0), 3) == 1.203


def test_planted_mistakes_are_caught():
    q, k, v = _qkv(4, 9, 3, seed=2)
    good = general.forward_head(q, k, v, True, 0.5, 3)
    ref = _brute(q, k, v, True, 0.5, 3)
    np.testing.assert_allclose(good[0], ref[0], rtol=1e-12, atol=1e-12)
    # window off by one (keys p - W <= j instead of p - W < j)
    bad = _brute(q, k, v, True, 0.5, 4)
    assert np.abs(good[0] - bad[0]).max() > 1e-3
    # causal aligned to the top-left instead of the bottom-right
    bad2 = general.forward_head(q, k[:4], v[:4], True, 0.5, 3)
    assert np.abs(good[0] - bad2[0]).max() > 1e-3


@pytest.mark.parametrize("nq,nk,d,dv,causal,window", [
    (5, 5, 3, 5, True, 0), (4, 9, 5, 2, True, 0), (6, 6, 4, 7, True, 2), (3, 8, 2, 6, False, 0),
])
def test_value_head_size_differs_from_key_head_size(nq, nk, d, dv, causal, window):
    q, k, v = _qkv(nq, nk, d, dv=dv, seed=nq * 13 + nk + dv)
    o, lse = general.forward_head(q, k, v, causal, 0.55, window)
    assert o.shape == (nq, dv)
    ob, lb = _brute(q, k, v, causal, 0.55, window)
    np.testing.assert_allclose(o, ob, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lb, rtol=1e-12, atol=1e-12)
    if nq == nk:
        do = np.random.default_rng(4).standard_normal((nq, dv))
        g = general.backward_head(q, k, v, o, lse, do, causal, 0.55, window)
        assert g[0].shape == (nq, d) and g[1].shape == (nk, d) and g[2].shape == (nk, dv)
        n = finite_diff.gradients_general(q, k, v, do, causal, 0.55, window)
        for a, b in zip(g, n):
            np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-7)
