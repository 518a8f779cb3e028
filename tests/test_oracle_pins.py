"""Pins for the float64 CPU oracle (no GPU).

Each check fixes the oracle against something other than itself: values the
pages print, the pages' own tiled-versus-dense check, closed forms, textbook
special cases, library routines (scipy ``logsumexp``, PyTorch's float64 CPU
``scaled_dot_product_attention`` and autograd) and central finite
differences. The last group plants mistakes in copies of the oracle and
checks that a pin catches each one.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import dense, finite_diff, tiled

from conftest import GOLDEN


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand(n, d, seed, dv=None):
    r = np.random.default_rng(seed)
    return r.standard_normal((n, d)), r.standard_normal((n, d)), r.standard_normal((n, dv or d))


# --------------------------------------------------------------------------
# Checks. Each takes the oracle functions it exercises, so that the
# planted-mistake tests at the bottom can hand in a broken copy.
# --------------------------------------------------------------------------

def check_running_sum(running_stats):
    g = _load("running_sum.json")
    got = running_stats(g["blocks"])
    for (m, l), want in zip(got, g["after_block"]):
        assert m == want["m"]
        assert round(l, g["printed_decimals"]) == want["l"], (l, want["l"])


def check_explorer(tiled_head, dense_head):
    g = _load("explorer_fixture.json")
    q, k, v = (np.array(g[x], dtype=np.float64) for x in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(q.shape[1])
    o_ref, lse_ref = dense_head(q, k, v, False, scale)
    for kb in g["key_blocks"]:
        o, lse = tiled_head(q, k, v, False, scale, g["query_block"], kb)
        np.testing.assert_allclose(o, o_ref, rtol=g["rtol"], atol=g["atol"])
        np.testing.assert_allclose(lse, lse_ref, rtol=g["rtol"], atol=g["atol"])


def check_against_torch_forward(dense_head, causal, seed=3):
    q, k, v = _rand(37, 16, seed)
    scale = 0.37
    o, lse = dense_head(q, k, v, causal, scale)
    tq, tk, tv = (torch.from_numpy(x)[None, None] for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    np.testing.assert_allclose(o, ref[0, 0].numpy(), rtol=1e-12, atol=1e-12)
    s = scale * (tq @ tk.transpose(-1, -2))
    if causal:
        s = s.masked_fill(torch.ones(37, 37, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1)[0, 0].numpy(), rtol=1e-12, atol=1e-12)


def check_against_torch_backward(dense_head, backward_head, causal, seed=4):
    q, k, v = _rand(29, 8, seed)
    do = np.random.default_rng(seed + 100).standard_normal((29, 8))
    scale = 0.41
    o, lse = dense_head(q, k, v, causal, scale)
    dq, dk, dv = backward_head(q, k, v, o, lse, do, causal, scale)
    tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], is_causal=causal, scale=scale)
    (out[0, 0] * torch.from_numpy(do)).sum().backward()
    for mine, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        np.testing.assert_allclose(mine, ref.numpy(), rtol=1e-10, atol=1e-12)


def check_finite_differences(dense_head, backward_head, causal, seed=5):
    n, d = 6, 3
    q, k, v = _rand(n, d, seed)
    do = np.random.default_rng(seed + 7).standard_normal((n, d))
    scale = 0.8
    o, lse = dense_head(q, k, v, causal, scale)
    got = backward_head(q, k, v, o, lse, do, causal, scale)
    num = finite_diff.gradients(q, k, v, do, causal, scale, h=1e-6)
    for a, b in zip(got, num):
        err = np.abs(a - b).max() / max(np.abs(b).max(), 1e-30)
        assert err < 1e-6, err


def check_causal_first_row(dense_head):
    g = _load("explorer_fixture.json")
    q, k, v = (np.array(g[x], dtype=np.float64) for x in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(2)
    o, lse = dense_head(q, k, v, True, scale)
    # Row 0 of a lower-triangular mask sees only key 0: O_0 = v_0, LSE_0 = s_00.
    np.testing.assert_allclose(o[0], v[0], atol=1e-15)
    assert abs(lse[0] - scale * float(q[0] @ k[0])) < 1e-15
    # The last row sees every key: causal and full attention agree there.
    o_full, lse_full = dense_head(q, k, v, False, scale)
    np.testing.assert_allclose(o[-1], o_full[-1], atol=1e-15)
    assert abs(lse[-1] - lse_full[-1]) < 1e-15
    # and row 1 sees keys 0, 1 only: a two-term softmax
    s = scale * np.array([q[1] @ k[0], q[1] @ k[1]])
    w = 1.0 / (1.0 + math.exp(s[0] - s[1]))            # weight of key 1
    np.testing.assert_allclose(o[1], (1 - w) * v[0] + w * v[1], atol=1e-15)


# --------------------------------------------------------------------------
# Tests on the oracle as it stands.
# --------------------------------------------------------------------------

def test_running_sum_page_example():
    check_running_sum(tiled.running_stats)


def test_running_sum_matches_dense_lse():
    # the same row as a one-dimensional attention problem: scores 1, 3, 2, 5
    q = np.array([[1.0]])
    k = np.array([[1.0], [3.0], [2.0], [5.0]])
    v = np.zeros((4, 1))
    _, lse = dense.forward_head(q, k, v, False, 1.0)
    m, l = tiled.running_stats([[1, 3], [2, 5]])[-1]
    assert abs((m + math.log(l)) - lse[0]) < 1e-15


def test_explorer_tiled_equals_dense():
    check_explorer(tiled.attention_head, dense.forward_head)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,qb,kb", [(37, 8, 5), (130, 128, 128), (1, 2, 7), (64, 16, 64), (9, 4, 3)])
def test_tiled_equals_dense_ragged(causal, n, qb, kb):
    q, k, v = _rand(n, 4, seed=n + qb, dv=3)
    o_ref, lse_ref = dense.forward_head(q, k, v, causal, 0.7)
    o, lse = tiled.attention_head(q, k, v, causal, 0.7, qb, kb)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_rows_sum_to_one(causal):
    q, k, _ = _rand(33, 8, seed=11)
    p = dense.probabilities(q, k, causal, 0.5)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
    assert (p >= 0).all()
    if causal:
        assert np.all(p[np.triu_indices(33, 1)] == 0.0)


def test_causal_first_row_closed_form():
    check_causal_first_row(dense.forward_head)


@pytest.mark.parametrize("causal", [False, True])
def test_special_cases(causal):
    r = np.random.default_rng(21)
    n, d = 12, 5
    q, k, v = r.standard_normal((n, d)), r.standard_normal((n, d)), r.standard_normal((n, d))
    # one key: the output is that key's value, LSE its score
    o, lse = dense.forward_head(q[:1], k[:1], v[:1], causal, 0.3)
    np.testing.assert_allclose(o[0], v[0], atol=1e-15)
    assert abs(lse[0] - 0.3 * float(q[0] @ k[0])) < 1e-14
    # all keys equal: uniform weights -> mean of V (prefix mean under the mask)
    kk = np.repeat(k[:1], n, axis=0)
    o, lse = dense.forward_head(q, kk, v, causal, 0.3)
    counts = np.arange(1, n + 1)[:, None]
    want = np.cumsum(v, axis=0) / counts if causal else np.repeat(v.mean(0, keepdims=True), n, 0)
    np.testing.assert_allclose(o, want, atol=1e-13)
    s0 = 0.3 * (q @ k[0])
    want_lse = s0 + np.log(np.arange(1, n + 1) if causal else np.full(n, n))
    np.testing.assert_allclose(lse, want_lse, atol=1e-13)
    # scale 0: uniform average as well
    o, _ = dense.forward_head(q, k, v, causal, 0.0)
    np.testing.assert_allclose(o, want, atol=1e-13)
    # constant values: the output is that constant
    o, _ = dense.forward_head(q, k, np.full((n, d), 2.5), causal, 0.3)
    np.testing.assert_allclose(o, 2.5, atol=1e-14)
    # LSE equals a library log-sum-exp of the masked scaled scores
    from scipy.special import logsumexp
    s = 0.3 * (q @ k.T)
    if causal:
        s[np.triu_indices(n, 1)] = -np.inf
    _, lse = dense.forward_head(q, k, v, causal, 0.3)
    np.testing.assert_allclose(lse, logsumexp(s, axis=1), atol=1e-13)


def test_permutation_and_shift_invariance():
    r = np.random.default_rng(22)
    n, d = 17, 6
    q, k, v = r.standard_normal((n, d)), r.standard_normal((n, d)), r.standard_normal((n, d))
    o, lse = dense.forward_head(q, k, v, False, 0.4)
    perm = r.permutation(n)
    o2, lse2 = dense.forward_head(q, k[perm], v[perm], False, 0.4)
    np.testing.assert_allclose(o2, o, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, atol=1e-13)
    # adding c to every key adds scale * q_i . c to row i's scores: O unchanged
    c = r.standard_normal(d)
    for causal in (False, True):
        o, lse = dense.forward_head(q, k, v, causal, 0.4)
        o3, lse3 = dense.forward_head(q, k + c, v, causal, 0.4)
        np.testing.assert_allclose(o3, o, atol=1e-12)
        np.testing.assert_allclose(lse3, lse + 0.4 * (q @ c), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_against_torch(causal):
    check_against_torch_forward(dense.forward_head, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_against_torch(causal):
    check_against_torch_backward(dense.forward_head, dense.backward_head, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_finite_differences(causal):
    check_finite_differences(dense.forward_head, dense.backward_head, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_invariants(causal):
    q, k, v = _rand(23, 7, seed=31)
    do = np.random.default_rng(32).standard_normal((23, 7))
    o, lse = dense.forward_head(q, k, v, causal, 0.6)
    dq, dk, dv, parts = dense.backward_head(q, k, v, o, lse, do, causal, 0.6, return_parts=True)
    # rows of dS sum to zero because sum_j P_ij dP_ij = D_i
    np.testing.assert_allclose(parts["ds_rowsum"], 0.0, atol=1e-12)
    # hence the key gradients sum to zero
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
    # rows of P sum to one, so the value gradients sum to the output gradients
    np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), atol=1e-12)


def test_row_chunking_does_not_change_results(monkeypatch):
    q, k, v = _rand(50, 4, seed=41)
    do = np.random.default_rng(42).standard_normal((50, 4))
    for causal in (False, True):
        o, lse = dense.forward_head(q, k, v, causal, 0.5)
        g = dense.backward_head(q, k, v, o, lse, do, causal, 0.5)
        monkeypatch.setattr(dense, "ROW_CHUNK", 7)
        o2, lse2 = dense.forward_head(q, k, v, causal, 0.5)
        g2 = dense.backward_head(q, k, v, o, lse, do, causal, 0.5)
        monkeypatch.setattr(dense, "ROW_CHUNK", 512)
        np.testing.assert_allclose(o2, o, atol=1e-14)
        np.testing.assert_allclose(lse2, lse, atol=1e-14)
        for a, b in zip(g, g2):
            np.testing.assert_allclose(a, b, atol=1e-13)


def test_batched_wrappers_and_head_sampling():
    import synthetic_inputs as si
    x = si.make_small(2, 3, 20, 8, seed=7)
    o, lse = dense.forward(x["q"], x["k"], x["v"], True, 0.35)
    ot, lset = tiled.attention(x["q"], x["k"], x["v"], True, 0.35, 8, 6)
    np.testing.assert_allclose(o, ot, atol=1e-12)
    np.testing.assert_allclose(lse, lset, atol=1e-12)
    o2, lse2 = dense.forward(x["q"], x["k"], x["v"], True, 0.35, heads=[(1, 2)])
    np.testing.assert_allclose(o2[1, 2], o[1, 2], atol=0)
    assert np.isnan(o2[0, 0]).all()
    dq, dk, dv = dense.backward(x["q"], x["k"], x["v"], o, lse, x["do"], True, 0.35)
    for b in range(2):
        for h in range(3):
            g = dense.backward_head(x["q"][b, h], x["k"][b, h], x["v"][b, h], o[b, h], lse[b, h],
                                    x["do"][b, h], True, 0.35)
            np.testing.assert_allclose(dq[b, h], g[0], atol=0)


# --------------------------------------------------------------------------
# Planted mistakes: a broken copy of each oracle function must fail a pin.
# --------------------------------------------------------------------------

def _tiled_without_rescale(q, k, v, causal, scale, qb, kb):
    """The tiled recurrence with alpha dropped (old sums never rescaled)."""
    orig = tiled._tile_update

    def broken(m, l, a, t, v_tile):
        m_new, _, _ = orig(m, l, a, t, v_tile)
        ref = np.where(np.isfinite(m_new), m_new, 0.0)
        p = np.exp(t - ref[:, None])
        a_new = a + (p @ v_tile if v_tile is not None else 0)
        return m_new, l + p.sum(axis=1), a_new

    tiled._tile_update = broken
    try:
        return tiled.attention_head(q, k, v, causal, scale, qb, kb)
    finally:
        tiled._tile_update = orig


def _running_stats_without_rescale(blocks):
    orig = tiled._tile_update

    def broken(m, l, a, t, v_tile):
        m_new, _, a_new = orig(m, l, a, t, v_tile)
        ref = np.where(np.isfinite(m_new), m_new, 0.0)
        return m_new, l + np.exp(t - ref[:, None]).sum(axis=1), a_new

    tiled._tile_update = broken
    try:
        return tiled.running_stats(blocks)
    finally:
        tiled._tile_update = orig


def _dense_keys_misaligned(q, k, v, causal, scale):
    """Key rows indexed in reverse while value rows are not (an index mistake)."""
    return dense.forward_head(q, k[::-1], v, causal, scale)


def _dense_mask_flipped(q, k, v, causal, scale):
    """Causal mask on the wrong side of the diagonal."""
    if not causal:
        return dense.forward_head(q, k, v, causal, scale)
    o, lse = dense.forward_head(q[::-1], k[::-1], v[::-1], True, scale)
    return o[::-1], lse[::-1]


def _dense_scale_twice(q, k, v, causal, scale):
    return dense.forward_head(q, k, v, causal, scale * scale)


def _backward_sign_flip(q, k, v, o, lse, do, causal, scale):
    dq, dk, dv = dense.backward_head(q, k, v, o, lse, do, causal, scale)
    return dq, -dk, dv


def _backward_no_D(q, k, v, o, lse, do, causal, scale):
    """dS = P * dP, the rowsum(dO * O) term dropped."""
    zero_o = np.zeros_like(np.asarray(o, dtype=np.float64))
    return dense.backward_head(q, k, v, zero_o, lse, do, causal, scale)


def _backward_swap_dq_dk(q, k, v, o, lse, do, causal, scale):
    dq, dk, dv = dense.backward_head(q, k, v, o, lse, do, causal, scale)
    return dk, dq, dv


@pytest.mark.parametrize("case", [
    ("running sum, alpha dropped", lambda: check_running_sum(_running_stats_without_rescale)),
    ("tiled, alpha dropped", lambda: check_explorer(_tiled_without_rescale, dense.forward_head)),
    ("dense, keys misaligned", lambda: check_explorer(tiled.attention_head, _dense_keys_misaligned)),
    ("dense, mask flipped", lambda: check_causal_first_row(_dense_mask_flipped)),
    ("dense, scale squared", lambda: check_against_torch_forward(_dense_scale_twice, False)),
    ("backward, dK sign", lambda: check_finite_differences(dense.forward_head, _backward_sign_flip, False)),
    ("backward, D dropped", lambda: check_finite_differences(dense.forward_head, _backward_no_D, True)),
    ("backward, dQ/dK swapped", lambda: check_against_torch_backward(dense.forward_head, _backward_swap_dq_dk, True)),
], ids=lambda c: c[0])
def test_planted_mistake_is_caught(case):
    _, run = case
    with pytest.raises(AssertionError):
        run()
