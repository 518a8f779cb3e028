"""Pins of the dropout oracle (CPU only).

The dropout arithmetic is pinned by its reduction to the dropout-free oracle,
by central finite differences of the masked forward, by the identity
D_i = sum_j P_ij dP_ij, and by the mean over many masks converging to the
dropout-free output; the generator by its kept fraction, byte uniformity,
avalanche and stream separation. Each check takes the oracle functions it
exercises, so that the planted-mistake tests at the bottom can hand in a
broken copy.
"""

import numpy as np
import pytest

from oracle import dense, dropout, finite_diff


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# --------------------------------------------------------------------------
# Checks
# --------------------------------------------------------------------------

def check_no_dropout_is_dense(fwd, bwd, causal):
    q, k, v, do = (_rand((37, 8), s) for s in range(4))
    mask = dropout.keep_mask(3, 37, 37, 0.0, seed=123, offset=7)
    assert mask.all()
    o, lse = fwd(q, k, v, mask, dropout.keep_probability(0.0), causal, 0.3)
    o_ref, lse_ref = dense.forward_head(q, k, v, causal, 0.3)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)
    g = bwd(q, k, v, o, lse, do, mask, 1.0, causal, 0.3)
    g_ref = dense.backward_head(q, k, v, o_ref, lse_ref, do, causal, 0.3)
    for a, b in zip(g, g_ref):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def check_finite_differences(fwd, bwd, causal):
    n, d = 6, 3
    q, k, v, do = (_rand((n, d), 10 + s) for s in range(4))
    mask = np.random.default_rng(5).random((n, n)) >= 0.4
    keep = 0.6

    def loss(a, b, c, g):
        o, _ = dropout.forward_head_masked(a, b, c, mask, keep, causal, 0.7)
        return float((o * g).sum())

    num = finite_diff._numeric(loss, q, k, v, do, 1e-6)
    o, lse = fwd(q, k, v, mask, keep, causal, 0.7)
    ana = bwd(q, k, v, o, lse, do, mask, keep, causal, 0.7)
    for a, b in zip(ana, num):
        np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-7)


def check_mean_over_masks(fwd, p=0.3, trials=3000):
    n, d = 12, 4
    q, k, v = (_rand((n, d), 30 + s) for s in range(3))
    keep = dropout.keep_probability(p)
    outs = np.stack([fwd(q, k, v, dropout.keep_mask(0, n, n, p, seed=77, offset=t), keep, False, 0.5)[0]
                     for t in range(trials)])
    o_ref, _ = dense.forward_head(q, k, v, False, 0.5)
    err = np.abs(outs.mean(axis=0) - o_ref)
    sem = outs.std(axis=0) / np.sqrt(trials)
    assert (err <= 5 * sem + 1e-12).all()


def check_kept_fraction(mask_fn, p):
    m = mask_fn(5, 1024, 1024, p, seed=2024, offset=3)
    keep = dropout.keep_probability(p)
    assert abs(m.mean() - keep) <= 6 * np.sqrt(keep * (1 - keep) / m.size)
    assert abs(keep - (1 - p)) <= 1 / 512  # t = round(256 p)


# --------------------------------------------------------------------------
# Pins
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_no_dropout_is_the_dense_oracle(causal):
    check_no_dropout_is_dense(dropout.forward_head_masked, dropout.backward_head_masked, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(causal):
    check_finite_differences(dropout.forward_head_masked, dropout.backward_head_masked, causal)


def test_row_vector_D_is_the_probability_weighted_dP():
    n, d = 20, 5
    q, k, v, do = (_rand((n, d), 20 + s) for s in range(4))
    mask = dropout.keep_mask(0, n, n, 0.25, seed=9, offset=1)
    keep = dropout.keep_probability(0.25)
    o, lse = dropout.forward_head_masked(q, k, v, mask, keep, True, 0.5)
    p = dense.probabilities(q, k, True, 0.5)
    dp = (do @ v.T) * mask / keep
    np.testing.assert_allclose((do * o).sum(axis=1), (p * dp).sum(axis=1), rtol=1e-12, atol=1e-12)


def test_mean_over_masks_is_the_dropout_free_output():
    check_mean_over_masks(dropout.forward_head_masked)


@pytest.mark.parametrize("p", [0.1, 0.25, 0.5, 0.9])
def test_kept_fraction(p):
    check_kept_fraction(dropout.keep_mask, p)


def test_bytes_are_uniform():
    b = dropout.keep_bytes(1, 1024, 1024, seed=1, offset=0).ravel()
    counts = np.bincount(b, minlength=256)
    expected = b.size / 256
    chi2 = ((counts - expected) ** 2 / expected).sum()
    assert abs(chi2 - 255) < 6 * np.sqrt(2 * 255)


def test_one_counter_bit_changes_half_the_output():
    rng = np.random.default_rng(3)
    n = 4000
    c = rng.integers(0, 2**32, size=(4, n), dtype=np.uint64)
    base = np.stack(dropout.philox4x32(*c, 0x12345678, 0x9ABCDEF0))
    word = rng.integers(0, 4, size=n)
    bit = rng.integers(0, 32, size=n).astype(np.uint64)
    c2 = c.copy()
    c2[word, np.arange(n)] ^= np.uint64(1) << bit
    flip = np.stack(dropout.philox4x32(*c2, 0x12345678, 0x9ABCDEF0))
    x = (base ^ flip).astype(np.uint32)
    bits = np.unpackbits(x.view(np.uint8)).reshape(-1).sum() / n
    assert 63.0 < bits < 65.0


def test_streams_are_separate():
    p = 0.5
    a = dropout.keep_mask(0, 64, 64, p, seed=1, offset=0)
    for other in (dropout.keep_mask(1, 64, 64, p, seed=1, offset=0),
                  dropout.keep_mask(0, 64, 64, p, seed=1, offset=1),
                  dropout.keep_mask(0, 64, 64, p, seed=2, offset=0),
                  dropout.keep_mask(0, 64, 64, p, seed=1 << 32, offset=0)):
        agree = (a == other).mean()
        assert 0.4 < agree < 0.6
    # a prefix of a longer head is the same mask (element (i, j) depends only on i, j)
    big = dropout.keep_mask(0, 100, 100, p, seed=1, offset=0)
    assert (big[:64, :64] == a).all()


# --------------------------------------------------------------------------
# Planted mistakes: a broken copy of each oracle function must fail a pin.
# --------------------------------------------------------------------------

def _bwd_dv_unmasked(q, k, v, o, lse, do, mask, keep, causal, scale):
    dq, dk, _ = dropout.backward_head_masked(q, k, v, o, lse, do, mask, keep, causal, scale)
    p = dense.probabilities(q, k, causal, scale)
    return dq, dk, p.T @ np.asarray(do, dtype=np.float64)


def _bwd_dp_not_rescaled(q, k, v, o, lse, do, mask, keep, causal, scale):
    """dP = (dO V^T) * M, the 1/keep left out (dV keeps it)."""
    _, _, dv = dropout.backward_head_masked(q, k, v, o, lse, do, mask, keep, causal, scale)
    dq, dk, _ = dropout.backward_head_masked(q, k, v, o, lse, do, mask, 1.0, causal, scale)
    return dq, dk, dv


def _bwd_D_without_dropout(q, k, v, o, lse, do, mask, keep, causal, scale):
    """D from the dropout-free O."""
    o_plain, _ = dense.forward_head(q, k, v, causal, scale)
    return dropout.backward_head_masked(q, k, v, o_plain, lse, do, mask, keep, causal, scale)


def _bwd_mask_transposed(q, k, v, o, lse, do, mask, keep, causal, scale):
    return dropout.backward_head_masked(q, k, v, o, lse, do, np.asarray(mask).T, keep, causal, scale)


def _fwd_not_rescaled(q, k, v, mask, keep, causal, scale):
    o, lse = dropout.forward_head_masked(q, k, v, mask, keep, causal, scale)
    return o * keep, lse


def _mask_threshold_off_by_one(bh, nq, nk, p, seed, offset):
    return dropout.keep_bytes(bh, nq, nk, seed, offset) > dropout.threshold(p)


@pytest.mark.parametrize("case", [
    ("backward, dV unmasked",
     lambda: check_finite_differences(dropout.forward_head_masked, _bwd_dv_unmasked, False)),
    ("backward, dP without 1/keep",
     lambda: check_finite_differences(dropout.forward_head_masked, _bwd_dp_not_rescaled, True)),
    ("backward, D from the dropout-free O",
     lambda: check_finite_differences(dropout.forward_head_masked, _bwd_D_without_dropout, False)),
    ("backward, mask transposed",
     lambda: check_finite_differences(dropout.forward_head_masked, _bwd_mask_transposed, False)),
    ("forward, 1/keep left out", lambda: check_mean_over_masks(_fwd_not_rescaled)),
    ("mask, keep test off by one", lambda: check_kept_fraction(_mask_threshold_off_by_one, 0.1)),
], ids=lambda c: c[0])
def test_planted_mistake_is_caught(case):
    _, run = case
    with pytest.raises(AssertionError):
        run()
