"""Attention with dropout on the probabilities -- TEST INFRASTRUCTURE.

Only tests, ``smoke()`` and ``bench.py``'s CPU legs use this module.

The pages name dropout once, as one of the settings to hold equal when
comparing attention implementations ("Flash Attention: IO-Aware Exact
Attention", section "What changes in FlashAttention-2"). They fix neither
where it applies nor how the mask is drawn. Reading taken here: inverted
dropout on the attention probabilities, the mask drawn from a counter-based
generator so that the backward regenerates exactly the forward's mask:

    P      = softmax of the (masked) scores, as in ``oracle.dense``
    M_ij   = 1 if byte_ij >= t else 0     (byte_ij from the generator below)
    keep   = (256 - t) / 256,  t = round(256 p) clamped to [0, 255]
    O      = (P * M) V / keep             LSE is the softmax statistic, unchanged

The backward of L = sum(O * dO), by calculus from that definition:

    dV = (P * M / keep)^T dO
    dP = (dO V^T) * M / keep
    D_i = sum_c dO_ic O_ic   (equal to sum_j P_ij dP_ij)
    dS = P * (dP - D 1^T)
    dQ = scale dS K,  dK = scale dS^T Q

Generator: Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random
numbers: as easy as 1, 2, 3", SC 2011), restated from its definition: a
counter of four 32-bit words and a key of two; each of ten rounds forms the
full 64-bit products of counter words 0 and 2 with the multipliers
0xD2511F53 and 0xCD9E8D57 and replaces the counter by
(hi(w2 product) ^ c1 ^ k0, lo(w2 product), hi(w0 product) ^ c3 ^ k1,
lo(w0 product)); the key grows by the Weyl increments (0x9E3779B9,
0xBB67AE85) before every round after the first.

Mask layout (the build's choice, so that both the forward, where a thread
owns a query row, and the backward, where a thread owns a key row, spend one
generator call per four elements): for batch-head index bh, query i, key j,

    counter = (j >> 2, i >> 2, bh, offset mod 2^32),  key = (seed mod 2^32, seed >> 32)
    byte_ij = byte (j & 3) (least significant first) of output word (i & 3)

so one call covers a 4 x 4 block of (query, key) pairs.

Pins (``tests/test_oracle_dropout.py``): p = 0 reduces to ``oracle.dense``;
central finite differences of the masked forward pin the backward; the mean
of O over many generator offsets converges to the dropout-free O (pins the
1/keep scale and the mask's independence from the data); the kept fraction
matches keep; the bytes are uniform and one flipped counter bit changes about
half of the output bits. The generator itself (``tests/test_oracle_philox.py``)
is pinned to Triton's independent Philox4x32, run on the CPU through its
interpreter, word for word at 1, 2, 7 and 10 rounds over edge and random
counters and keys, and its two key increments to their closed forms (the
first 32 fractional bits of the golden ratio and of sqrt(3)); near misses
(swapped multipliers, a wrong increment, exchanged product halves, an early
key bump, permuted words) each fail that pin.
"""

from __future__ import annotations

import numpy as np

from .dense import as_f64, scores

_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = np.uint64(0x9E3779B9)
_W1 = np.uint64(0xBB67AE85)
_MASK32 = np.uint64(0xFFFFFFFF)
ROUNDS = 10


def threshold(p: float) -> int:
    """The byte threshold t: an element is kept when its byte is >= t."""
    if not (0.0 <= p < 1.0):
        raise ValueError("dropout probability must be in [0, 1)")
    return int(min(255, max(0, round(256.0 * p))))


def keep_probability(p: float) -> float:
    return (256 - threshold(p)) / 256.0


def philox4x32(c0, c1, c2, c3, k0: int, k1: int, rounds: int = ROUNDS):
    """Philox4x32 on arrays of counter words (any common shape); returns four uint32 arrays."""
    c = [np.asarray(x, dtype=np.uint64) & _MASK32 for x in (c0, c1, c2, c3)]
    c = list(np.broadcast_arrays(*c))
    key0 = np.uint64(k0 & 0xFFFFFFFF)
    key1 = np.uint64(k1 & 0xFFFFFFFF)
    for r in range(rounds):
        if r > 0:
            key0 = (key0 + _W0) & _MASK32
            key1 = (key1 + _W1) & _MASK32
        p0 = c[0] * _M0  # < 2^64: exact in uint64
        p1 = c[2] * _M1
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c = [hi1 ^ c[1] ^ key0, lo1, hi0 ^ c[3] ^ key1, lo0]
    return tuple(x.astype(np.uint32) for x in c)


def keep_bytes(bh: int, nq: int, nk: int, seed: int, offset: int) -> np.ndarray:
    """byte_ij for queries [0, nq) and keys [0, nk) of batch-head ``bh`` (uint8 [nq, nk])."""
    qb = np.arange((nq + 3) // 4, dtype=np.uint64)[:, None]
    kb = np.arange((nk + 3) // 4, dtype=np.uint64)[None, :]
    w = philox4x32(kb, qb, np.uint64(bh), np.uint64(offset & 0xFFFFFFFF),
                   seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    words = np.stack(w, axis=0)  # [4 (query within block), nq/4, nk/4]
    out = np.empty((words.shape[1] * 4, words.shape[2] * 4), dtype=np.uint8)
    for qi in range(4):
        for kj in range(4):
            out[qi::4, kj::4] = ((words[qi] >> np.uint32(8 * kj)) & np.uint32(0xFF)).astype(np.uint8)
    return out[:nq, :nk]


def keep_mask(bh: int, nq: int, nk: int, p: float, seed: int, offset: int) -> np.ndarray:
    """M_ij (bool [nq, nk]) of batch-head ``bh``."""
    return keep_bytes(bh, nq, nk, seed, offset) >= threshold(p)


def forward_head_masked(q, k, v, mask, keep: float, causal: bool, scale: float):
    """O [N, d_v] and LSE [N] of one head with a given keep mask and keep probability."""
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    s = scores(q, k, causal, scale)
    m = s.max(axis=1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe)
    l = e.sum(axis=1, keepdims=True)
    ok = l[:, 0] > 0
    p = np.where(l > 0, e / np.where(l > 0, l, 1.0), 0.0)
    o = ((p * mask) @ v) / keep
    o[~ok] = 0.0
    with np.errstate(divide="ignore"):
        lse = np.where(ok, m_safe[:, 0] + np.log(np.where(ok, l[:, 0], 1.0)), -np.inf)
    return o, lse


def backward_head_masked(q, k, v, o, lse, do, mask, keep: float, causal: bool, scale: float):
    """dQ, dK, dV of one head with a given keep mask (see the module docstring)."""
    q, k, v, o, do = (as_f64(t) for t in (q, k, v, o, do))
    lse = as_f64(lse)
    s = scores(q, k, causal, scale)
    lse_c = lse[:, None]
    lse_safe = np.where(np.isfinite(lse_c), lse_c, 0.0)
    p = np.where(np.isfinite(lse_c), np.exp(s - lse_safe), 0.0)
    pd = p * mask / keep
    dv = pd.T @ do
    dp = (do @ v.T) * mask / keep
    D = (do * o).sum(axis=1)
    ds = p * (dp - D[:, None])
    return scale * (ds @ k), scale * (ds.T @ q), dv


def forward(q, k, v, causal: bool, scale: float, p: float, seed: int, offset: int, heads=None):
    """Batched [B, H, N, d] dropout forward; heads not listed stay NaN."""
    B, H, N = q.shape[0], q.shape[1], q.shape[2]
    o = np.full((B, H, N, v.shape[3]), np.nan)
    lse = np.full((B, H, N), np.nan)
    keep = keep_probability(p)
    for b, h in (heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]):
        mask = keep_mask(b * H + h, N, k.shape[2], p, seed, offset)
        o[b, h], lse[b, h] = forward_head_masked(q[b, h], k[b, h], v[b, h], mask, keep, causal, scale)
    return o, lse


def backward(q, k, v, o, lse, do, causal: bool, scale: float, p: float, seed: int, offset: int,
             heads=None):
    """Batched dropout backward; ``o`` and ``lse`` are the oracle's own forward results."""
    B, H, N = q.shape[0], q.shape[1], q.shape[2]
    dq = np.full(tuple(q.shape), np.nan)
    dk = np.full(tuple(k.shape), np.nan)
    dv = np.full(tuple(v.shape), np.nan)
    keep = keep_probability(p)
    for b, h in (heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]):
        mask = keep_mask(b * H + h, N, k.shape[2], p, seed, offset)
        dq[b, h], dk[b, h], dv[b, h] = backward_head_masked(
            q[b, h], k[b, h], v[b, h], o[b, h], lse[b, h], do[b, h], mask, keep, causal, scale)
    return dq, dk, dv
