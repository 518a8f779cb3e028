"""Merging partial softmax states of a split key range -- TEST INFRASTRUCTURE.

Only tests, ``smoke()`` and ``bench.py``'s CPU-baseline leg use this module.

"FlashAttention -- the same attention, made memory-aware", section 03
("Reconcile: merge each tile into the running answer"), combines the state
carried so far -- running maximum m_prev, denominator l_prev and the output
O_prev normalised by l_prev -- with a new tile's maximum m, denominator l
and unnormalised contribution pv:

    m_new = max(m_prev, m)
    l_new = exp(m_prev - m_new) * l_prev + exp(m - m_new) * l
    O_new = (l_prev * exp(m_prev - m_new) * O_prev + exp(m - m_new) * pv) / l_new

Nothing in the rule requires the new part to be one tile: a whole chunk of
keys, reduced on its own to (m, l, O) with pv = l * O, merges the same way,
so a key range split into chunks processed independently (decode over a long
key/value cache) is recombined by applying the rule chunk after chunk. A
part that saw no key has m = -inf and l = 0 and contributes nothing.

A part is handed in as (O, LSE) with LSE = m + ln(l) -- the statistic the
library saves -- and split back into m = LSE, l = 1 (the same state: only
the product exp(m) * l enters the result).

Pins: merging the parts of any split equals the unsplit ``general``
forward; the order of merging does not matter; the worked running sum of
"FlashAttention" (Road to Intelligence), section "The trick that makes
tiling possible" -- scores [1, 3] then [2, 5] -- merged as two parts gives
the page's l = 1.203 against the final maximum 5 (``tests/test_oracle_general.py``).
"""

from __future__ import annotations

import numpy as np


def merge_two(m_prev, l_prev, o_prev, m, l, o):
    """The section-03 rule for arrays of rows: returns (m_new, l_new, O_new)."""
    m_new = np.maximum(m_prev, m)
    ref = np.where(np.isfinite(m_new), m_new, 0.0)
    a_prev = np.where(np.isfinite(m_prev), np.exp(m_prev - ref), 0.0)
    a = np.where(np.isfinite(m), np.exp(m - ref), 0.0)
    l_new = a_prev * l_prev + a * l
    pv = l[..., None] * o                      # the part's unnormalised P V
    num = (l_prev * a_prev)[..., None] * o_prev + a[..., None] * pv
    with np.errstate(invalid="ignore", divide="ignore"):
        o_new = np.where(l_new[..., None] > 0, num / np.where(l_new > 0, l_new, 1.0)[..., None], 0.0)
    return m_new, l_new, o_new


def merge(parts):
    """Merge a list of (O [rows, d_v], LSE [rows]) parts, first to last.

    Returns (O, LSE) of the union of the parts' keys.
    """
    o0, lse0 = parts[0]
    rows, dv = np.asarray(o0).shape
    m = np.full(rows, -np.inf)
    l = np.zeros(rows)
    o = np.zeros((rows, dv))
    for o_p, lse_p in parts:
        lse_p = np.asarray(lse_p, dtype=np.float64)
        l_p = np.where(np.isfinite(lse_p), 1.0, 0.0)
        m, l, o = merge_two(m, l, o, lse_p, l_p, np.asarray(o_p, dtype=np.float64))
    with np.errstate(divide="ignore"):
        lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return o, lse
