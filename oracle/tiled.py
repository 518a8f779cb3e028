"""Tiled online-softmax attention in float64 -- TEST INFRASTRUCTURE.

Only tests, ``smoke()`` and ``bench.py``'s CPU-baseline leg use this module.

A literal restatement of the forward recurrence of "Flash Attention: IO-Aware
Exact Attention" (sections "Online softmax makes tiling exact", "Loop order
changes which data is reloaded" and "Check the recurrence on CPU"): the
query-block-outer, key-block-inner order, where one block of queries and its
row state stay resident while every key/value block passes. Per query row the
state is a running maximum m, a denominator l and an unnormalised numerator
a (a d_v-vector). It starts at m = -inf, l = 0, a = 0, and for each tile of
scores t with values V_tile:

    m'    = max(m, rowmax t)
    alpha = exp(m - m')            (alpha = 0 while no key has been seen)
    p     = exp(t - m')
    l     = alpha * l + rowsum p
    a     = alpha * a + p V_tile
    m     = m'

and after the last tile O = a / l, one division per row (the page's remark
that FlashAttention-2 keeps the numerator unnormalised). The page names
causal masks and tail blocks without showing them; here a causal mask sets
t = -inf where key j > query i, and tail blocks are simply shorter slices.
The log-sum-exp LSE = m + ln(l) is returned as the saved statistic.

Where a whole tile row is masked and m' is still -inf, p and alpha are taken
as 0 (the page defines alpha = 0 before any key is seen); the row state then
does not change.

``running_stats`` is the same update restricted to (m, l) for one row of
scores handed in block by block -- the worked example of "FlashAttention"
(Road to Intelligence), section "The trick that makes tiling possible".

Pins: the page's explorer fixture with key tiles 1, 2, 3, 4 and 7 against
``dense`` (rtol = atol = 1e-12, as on the page); the worked running sum
(l = 1.135 after [1, 3], l = 1.203 after [2, 5]); random ragged and causal
cases against ``dense``.
"""

from __future__ import annotations

import numpy as np



def as_f64(x) -> np.ndarray:
    """Exact upcast of a numpy array or a (CPU) torch tensor to float64."""
    if isinstance(x, np.ndarray):
        return x.astype(np.float64, copy=False)
    return x.detach().to("cpu").float().numpy().astype(np.float64)


def _tile_update(m, l, a, t, v_tile):
    """One step of the recurrence for a block of rows. Returns (m', l', a')."""
    m_new = np.maximum(m, t.max(axis=1))
    seen = np.isfinite(m_new)
    m_ref = np.where(seen, m_new, 0.0)            # finite stand-in for m' = -inf
    alpha = np.where(np.isfinite(m), np.exp(m - m_ref), 0.0)
    p = np.where(seen[:, None], np.exp(t - m_ref[:, None]), 0.0)
    l_new = alpha * l + p.sum(axis=1)
    a_new = alpha[:, None] * a
    if v_tile is not None:
        a_new = a_new + p @ v_tile
    return m_new, l_new, a_new


def running_stats(score_blocks):
    """(m, l) of one row of scores after each block, via the recurrence."""
    m = np.full(1, -np.inf)
    l = np.zeros(1)
    a = np.zeros((1, 0))
    out = []
    for blk in score_blocks:
        t = np.asarray(blk, dtype=np.float64)[None, :]
        m, l, a = _tile_update(m, l, a, t, None)
        out.append((float(m[0]), float(l[0])))
    return out


def attention_head(q, k, v, causal: bool = False, scale: float | None = None,
                   query_block: int = 2, key_block: int = 2):
    """O [N, d_v] and LSE [N] of one head by the tiled recurrence."""
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    if scale is None:
        scale = 1.0 / np.sqrt(q.shape[1])
    n_q, n_k = q.shape[0], k.shape[0]
    out = np.empty((n_q, v.shape[1]), dtype=np.float64)
    lse = np.empty(n_q, dtype=np.float64)
    for row in range(0, n_q, query_block):
        query = q[row:row + query_block]
        rows = np.arange(row, row + len(query))
        m = np.full(len(query), -np.inf)
        l = np.zeros(len(query))
        a = np.zeros((len(query), v.shape[1]))
        for col in range(0, n_k, key_block):
            keys = k[col:col + key_block]
            t = (query @ keys.T) * scale
            if causal:
                cols = np.arange(col, col + len(keys))
                t = np.where(cols[None, :] > rows[:, None], -np.inf, t)
            m, l, a = _tile_update(m, l, a, t, v[col:col + key_block])
        ok = l > 0
        with np.errstate(invalid="ignore", divide="ignore"):
            out[row:row + len(query)] = np.where(ok[:, None], a / np.where(ok, l, 1.0)[:, None], 0.0)
            lse[row:row + len(query)] = np.where(ok, m + np.log(np.where(ok, l, 1.0)), -np.inf)
    return out, lse


def attention(q, k, v, causal: bool, scale: float, query_block: int = 128,
              key_block: int = 128):
    """Batched tiled forward over [B, H, N, d] inputs (float64 results)."""
    B, H, N = q.shape[0], q.shape[1], q.shape[2]
    o = np.empty((B, H, N, v.shape[3]))
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = attention_head(q[b, h], k[b, h], v[b, h], causal, scale,
                                                query_block, key_block)
    return o, lse
