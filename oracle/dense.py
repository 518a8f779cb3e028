"""Dense float64 attention: the definition written out -- TEST INFRASTRUCTURE.

Only tests, ``smoke()`` and ``bench.py``'s CPU-baseline leg use this module.

Forward, per head with i, j in [0, N) ("Flash Attention: IO-Aware Exact
Attention", section "Why intermediate matrices cost memory traffic", and the
dense check in section "Check the recurrence on CPU"; the scale and causal
mask as in the dense PyTorch block of "FlashAttention -- the same attention,
made memory-aware", section 00):

    s_ij  = scale * sum_c q_ic k_jc,   s_ij = -inf where causal and j > i
    m_i   = max_j s_ij
    l_i   = sum_j exp(s_ij - m_i)
    O_i   = sum_j exp(s_ij - m_i) v_j / l_i
    LSE_i = m_i + ln(l_i)          (the per-row normalisation statistic the
                                    forward saves for the backward, section
                                    "Storage, arithmetic and IO are separate
                                    quantities")

Backward: the gradients of L = sum(O * dO), obtained from the definition by
calculus (the pages state only that the backward recomputes scores from Q, K
and V instead of storing them):

    P  = exp(s - LSE)          dV = P^T dO          dP = dO V^T
    D_i = sum_c dO_ic O_ic     dS = P * (dP - D 1^T)
    dQ = scale * dS K          dK = scale * dS^T Q

A row with every key masked (impossible for a causal mask with as many keys
as queries, since the diagonal is visible) gets O = 0 and LSE = -inf.

Pins: the page's explorer fixture against ``tiled`` (an independent
restatement), rows of P summing to 1, the causal first-row closed form,
textbook special cases, scipy's ``logsumexp``, PyTorch's float64 CPU
``scaled_dot_product_attention`` and autograd, and central finite
differences (``finite_diff``).
"""

from __future__ import annotations

import numpy as np

ROW_CHUNK = 512


def as_f64(x) -> np.ndarray:
    """Exact upcast of a numpy array or a (CPU) torch tensor to float64."""
    if isinstance(x, np.ndarray):
        return x.astype(np.float64, copy=False)
    # torch tensor (bf16/fp16/fp32): via float32, which holds bf16 exactly
    return x.detach().to("cpu").float().numpy().astype(np.float64)


def scores(q: np.ndarray, k: np.ndarray, causal: bool, scale: float,
           row0: int = 0) -> np.ndarray:
    """s = scale * q k^T for query rows row0.. of one head, causal mask applied."""
    s = (q @ k.T) * scale
    if causal:
        rows = np.arange(row0, row0 + q.shape[0])[:, None]
        cols = np.arange(k.shape[0])[None, :]
        s = np.where(cols > rows, -np.inf, s)
    return s


def probabilities(q, k, causal: bool, scale: float) -> np.ndarray:
    """Row softmax of the (masked) scores of one head, as a full N x N matrix."""
    q, k = as_f64(q), as_f64(k)
    s = scores(q, k, causal, scale)
    m = s.max(axis=1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe)
    l = e.sum(axis=1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        p = np.where(l > 0, e / np.where(l > 0, l, 1.0), 0.0)
    return p


def forward_head(q, k, v, causal: bool, scale: float):
    """O [N, d_v] and LSE [N] of one head, in row chunks of ROW_CHUNK queries."""
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    n = q.shape[0]
    o = np.zeros((n, v.shape[1]), dtype=np.float64)
    lse = np.full(n, -np.inf, dtype=np.float64)
    for r0 in range(0, n, ROW_CHUNK):
        r1 = min(n, r0 + ROW_CHUNK)
        kk = k[:r1] if causal else k
        vv = v[:r1] if causal else v
        s = scores(q[r0:r1], kk, causal, scale, row0=r0)
        m = s.max(axis=1)
        m_safe = np.where(np.isfinite(m), m, 0.0)
        e = np.exp(s - m_safe[:, None])
        l = e.sum(axis=1)
        ok = l > 0
        o[r0:r1][ok] = (e[ok] @ vv) / l[ok, None]
        with np.errstate(divide="ignore"):
            lse[r0:r1] = np.where(ok, m_safe + np.log(np.where(ok, l, 1.0)), -np.inf)
    return o, lse


def backward_head(q, k, v, o, lse, do, causal: bool, scale: float,
                  return_parts: bool = False):
    """dQ, dK, dV of L = sum(O * dO) for one head (see the module docstring).

    ``o`` and ``lse`` are this head's forward results. With ``return_parts``
    the row vector D and the row sums of dS are returned too (for the
    invariant sum_j dS_ij = 0).
    """
    q, k, v, o, do = (as_f64(t) for t in (q, k, v, o, do))
    lse = as_f64(lse)
    n = q.shape[0]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    D = (do * o).sum(axis=1)
    ds_rowsum = np.zeros(n)
    for r0 in range(0, n, ROW_CHUNK):
        r1 = min(n, r0 + ROW_CHUNK)
        c1 = r1 if causal else k.shape[0]
        s = scores(q[r0:r1], k[:c1], causal, scale, row0=r0)
        lse_c = lse[r0:r1, None]
        lse_safe = np.where(np.isfinite(lse_c), lse_c, 0.0)
        p = np.where(np.isfinite(lse_c), np.exp(s - lse_safe), 0.0)
        dv[:c1] += p.T @ do[r0:r1]
        dp = do[r0:r1] @ v[:c1].T
        ds = p * (dp - D[r0:r1, None])
        ds_rowsum[r0:r1] = ds.sum(axis=1)
        dq[r0:r1] = scale * (ds @ k[:c1])
        dk[:c1] += scale * (ds.T @ q[r0:r1])
    if return_parts:
        return dq, dk, dv, {"D": D, "ds_rowsum": ds_rowsum}
    return dq, dk, dv


def _heads(shape, heads):
    B, H = shape[0], shape[1]
    if heads is None:
        return [(b, h) for b in range(B) for h in range(H)]
    return list(heads)


def forward(q, k, v, causal: bool, scale: float, heads=None):
    """Batched forward over [B, H, N, d] inputs.

    Returns (O [B,H,N,d_v], LSE [B,H,N]) in float64. With ``heads`` (a list
    of (b, h) pairs) only those heads are computed; the others stay NaN.
    """
    B, H, N = q.shape[0], q.shape[1], q.shape[2]
    dv_ = v.shape[3]
    o = np.full((B, H, N, dv_), np.nan)
    lse = np.full((B, H, N), np.nan)
    for b, h in _heads(q.shape, heads):
        o[b, h], lse[b, h] = forward_head(q[b, h], k[b, h], v[b, h], causal, scale)
    return o, lse


def backward(q, k, v, o, lse, do, causal: bool, scale: float, heads=None):
    """Batched backward; ``o`` and ``lse`` are the oracle's own forward results."""
    B, H = q.shape[0], q.shape[1]
    shape_q = tuple(q.shape)
    shape_v = tuple(v.shape)
    dq = np.full(shape_q, np.nan)
    dk = np.full(shape_q, np.nan)
    dv = np.full(shape_v, np.nan)
    for b, h in _heads((B, H), heads):
        dq[b, h], dk[b, h], dv[b, h] = backward_head(
            q[b, h], k[b, h], v[b, h], o[b, h], lse[b, h], do[b, h], causal, scale)
    return dq, dk, dv
