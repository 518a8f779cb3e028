"""Dense float64 attention with general masks -- TEST INFRASTRUCTURE.

Only tests, ``smoke()`` and ``bench.py``'s CPU-baseline leg use this module.

The definition of ``dense`` extended to the masks the library's extended
entry points take, for one head with Nq queries and Nk keys:

  * queries and keys may differ in number; with a causal mask the queries
    are the last Nq positions of the Nk keys (a decode step over a key/value
    cache: "Flash Attention: IO-Aware Exact Attention", section "What changes
    in FlashAttention-2", which names KV caching for decode-time history), so
    query i sits at position i + off with off = Nk - Nq and may see keys
    j <= i + off;
  * a sliding window of W >= 1 keys (same section: sliding-window attention
    changes which historical keys can participate) keeps, for a causal
    query at position p = i + off, only the keys p - W < j <= p.

    visible(i, j) = (not causal or j <= i + off) and (W == 0 or j > i + off - W)
    s_ij = scale * q_i . k_j   where visible, -inf elsewhere
    O_i  = sum_j exp(s_ij - m_i) v_j / l_i,   LSE_i = m_i + ln(l_i)

and, for the backward (training, Nq = Nk), the gradients of L = sum(O * dO)
with the same formulas as ``dense``. A row that sees no key has O = 0 and
LSE = -inf (it can happen only for a key range that excludes all of a row's
keys, as in one split of a split key range).

Pins: with Nq = Nk and no window the functions equal ``dense``; a brute-force
per-row evaluation over an explicit slice of visible keys (a different code
path from masking); window 1 gives O_i = v_{i+off} and LSE_i = s_{i,i+off};
a window at least Nk wide equals the plain causal mask; one decode query
with a causal mask sees every key; the backward against central finite
differences with offsets and windows (``tests/test_oracle_general.py``).
"""

from __future__ import annotations

import numpy as np

from .dense import as_f64


def visible(nq: int, nk: int, causal: bool, window: int) -> np.ndarray:
    """Boolean [nq, nk]: which keys each query may attend to."""
    off = nk - nq
    pos = np.arange(nq)[:, None] + off
    cols = np.arange(nk)[None, :]
    ok = np.ones((nq, nk), dtype=bool)
    if causal:
        ok &= cols <= pos
    if window:
        ok &= cols > pos - window
    return ok


def forward_head(q, k, v, causal: bool, scale: float, window: int = 0, key_range=None):
    """O [Nq, d_v] and LSE [Nq] of one head.

    ``key_range`` = (lo, hi) restricts the keys to lo <= j < hi (one split of
    a split key range); the mask keeps its meaning in absolute positions.
    """
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    nq, nk = q.shape[0], k.shape[0]
    s = (q @ k.T) * scale
    ok = visible(nq, nk, causal, window)
    if key_range is not None:
        lo, hi = key_range
        cols = np.arange(nk)[None, :]
        ok &= (cols >= lo) & (cols < hi)
    s = np.where(ok, s, -np.inf)
    m = s.max(axis=1)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.where(ok, np.exp(s - m_safe[:, None]), 0.0)
    l = e.sum(axis=1)
    live = l > 0
    o = np.zeros((nq, v.shape[1]))
    o[live] = (e[live] @ v) / l[live, None]
    with np.errstate(divide="ignore"):
        lse = np.where(live, m_safe + np.log(np.where(live, l, 1.0)), -np.inf)
    return o, lse


def backward_head(q, k, v, o, lse, do, causal: bool, scale: float, window: int = 0):
    """dQ, dK, dV of L = sum(O * dO) for one head with the general mask."""
    q, k, v, o, do = (as_f64(t) for t in (q, k, v, o, do))
    lse = as_f64(lse)
    nq, nk = q.shape[0], k.shape[0]
    ok = visible(nq, nk, causal, window)
    s = (q @ k.T) * scale
    lse_c = lse[:, None]
    live = np.isfinite(lse_c) & ok
    p = np.where(live, np.exp(np.where(live, s - np.where(np.isfinite(lse_c), lse_c, 0.0), 0.0)), 0.0)
    D = (do * o).sum(axis=1)
    dv = p.T @ do
    dp = do @ v.T
    ds = p * (dp - D[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv


def forward(q, k, v, causal: bool, scale: float, window: int = 0, heads=None):
    """Batched forward over [B, H, Nq, d] queries and [B, H, Nk, d] keys/values.

    Returns (O [B,H,Nq,d_v], LSE [B,H,Nq]) in float64; with ``heads`` only
    those (b, h) pairs are computed, the others stay NaN.
    """
    B, H, nq = q.shape[0], q.shape[1], q.shape[2]
    o = np.full((B, H, nq, v.shape[3]), np.nan)
    lse = np.full((B, H, nq), np.nan)
    pairs = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    for b, h in pairs:
        o[b, h], lse[b, h] = forward_head(q[b, h], k[b, h], v[b, h], causal, scale, window)
    return o, lse


def backward(q, k, v, o, lse, do, causal: bool, scale: float, window: int = 0, heads=None):
    """Batched backward with the general mask (o, lse: the oracle's forward)."""
    B, H = q.shape[0], q.shape[1]
    dq = np.full(tuple(q.shape), np.nan)
    dk = np.full(tuple(k.shape), np.nan)
    dv = np.full(tuple(v.shape), np.nan)
    pairs = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    for b, h in pairs:
        dq[b, h], dk[b, h], dv[b, h] = backward_head(q[b, h], k[b, h], v[b, h], o[b, h],
                                                     lse[b, h], do[b, h], causal, scale, window)
    return dq, dk, dv
