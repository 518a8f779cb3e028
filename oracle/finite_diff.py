"""Central finite differences for the attention backward -- TEST INFRASTRUCTURE.

Only tests use this module. It differentiates the scalar L = sum(O * dO),
where O is the dense forward of ``oracle.dense``, numerically: for every
input element x, dL/dx ~ (L(x + h) - L(x - h)) / (2 h). This pins the
analytic backward of ``oracle.dense`` (whose equations the pages do not give;
"FlashAttention" (Road to Intelligence), section "What to remember", says
only that the backward recomputes the scores from Q, K and V) to the
forward's own definition. Use tiny heads only (N <= 8, d <= 4).
``gradients_general`` does the same for the forward of ``oracle.general``
(queries over a longer key range, sliding windows).
"""

from __future__ import annotations

import numpy as np

from .dense import forward_head
from . import general


def loss(q, k, v, do, causal: bool, scale: float) -> float:
    o, _ = forward_head(q, k, v, causal, scale)
    return float((o * do).sum())


def _numeric(loss_fn, q, k, v, do, h):
    q, k, v, do = (np.array(t, dtype=np.float64) for t in (q, k, v, do))
    grads = []
    for target in (q, k, v):
        g = np.zeros_like(target)
        for idx in np.ndindex(target.shape):
            keep = target[idx]
            target[idx] = keep + h
            lp = loss_fn(q, k, v, do)
            target[idx] = keep - h
            lm = loss_fn(q, k, v, do)
            target[idx] = keep
            g[idx] = (lp - lm) / (2.0 * h)
        grads.append(g)
    return tuple(grads)


def gradients(q, k, v, do, causal: bool, scale: float, h: float = 1e-6):
    """Numerical (dQ, dK, dV) of L = sum(O * dO) for one head (float64)."""
    return _numeric(lambda a, b, c, d: loss(a, b, c, d, causal, scale), q, k, v, do, h)


def gradients_general(q, k, v, do, causal: bool, scale: float, window: int = 0, h: float = 1e-6):
    """Numerical (dQ, dK, dV) of L = sum(O * dO) with the general mask."""
    def lf(a, b, c, d):
        o, _ = general.forward_head(a, b, c, causal, scale, window)
        return float((o * d).sum())
    return _numeric(lf, q, k, v, do, h)
