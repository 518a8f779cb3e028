"""Central finite differences for the attention backward -- TEST INFRASTRUCTURE.

Only tests use this module. It differentiates the scalar L = sum(O * dO),
where O is the dense forward of ``oracle.dense``, numerically: for every
input element x, dL/dx ~ (L(x + h) - L(x - h)) / (2 h). This pins the
analytic backward of ``oracle.dense`` (whose equations the pages do not give;
"FlashAttention" (Road to Intelligence), section "What to remember", says
only that the backward recomputes the scores from Q, K and V) to the
forward's own definition. Use tiny heads only (N <= 8, d <= 4).
"""

from __future__ import annotations

import numpy as np

from .dense import forward_head


def loss(q, k, v, do, causal: bool, scale: float) -> float:
    o, _ = forward_head(q, k, v, causal, scale)
    return float((o * do).sum())


def gradients(q, k, v, do, causal: bool, scale: float, h: float = 1e-6):
    """Numerical (dQ, dK, dV) of L = sum(O * dO) for one head (float64)."""
    q, k, v, do = (np.array(t, dtype=np.float64) for t in (q, k, v, do))
    grads = []
    for target in (q, k, v):
        g = np.zeros_like(target)
        for idx in np.ndindex(target.shape):
            keep = target[idx]
            target[idx] = keep + h
            lp = loss(q, k, v, do, causal, scale)
            target[idx] = keep - h
            lm = loss(q, k, v, do, causal, scale)
            target[idx] = keep
            g[idx] = (lp - lm) / (2.0 * h)
        grads.append(g)
    return tuple(grads)
