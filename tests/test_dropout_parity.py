"""Dropout forward and backward on the GPU against the float64 oracle.

Two kinds of checks:
- the keep mask itself, bit for bit: with Q = 0 every visible probability
  is exactly 1/N, and one-hot rows of V (forward) or dO (backward) scaled by
  2^t make each output element an integer code sum_t M 2^t over four keys
  (forward, O) or four queries (backward, dV); the codes are decoded from
  the kernel's outputs and compared with the oracle's mask;
- O, LSE and the gradients on random inputs against ``oracle.dropout`` with
  the gates of the dropout-free tests (forward: max |O - O_ref| <= 2e-2, mean
  <= 2e-3, LSE max <= 1e-3; backward: max-norm relative error <= 5e-2).
"""

import math

import numpy as np
import pytest

import synthetic_inputs as si
from oracle import dropout

torch = pytest.importorskip("torch")
fa = pytest.importorskip("exact_io_aware_33_gb300")

pytestmark = pytest.mark.gpu

SEED = 0x1234_5678_9ABC_DEF0


def _codes_inputs(B, H, N, d, kind):
    """q = 0, k random; V (kind 'fwd') or dO (kind 'bwd') one-hot: row r has
    2^(r // d) in column r % d, so that four rows share a column."""
    assert N == 4 * d
    g = torch.Generator().manual_seed(N + d)
    q = torch.zeros(B, H, N, d, dtype=torch.bfloat16)
    k = torch.randn(B, H, N, d, generator=g).to(torch.bfloat16)
    onehot = torch.zeros(N, d)
    r = torch.arange(N)
    onehot[r, r % d] = (2.0 ** (r // d)).float()
    rnd = torch.randn(B, H, N, d, generator=g).to(torch.bfloat16)
    special = onehot.to(torch.bfloat16).expand(B, H, N, d).contiguous()
    v = special if kind == "fwd" else rnd
    do = special if kind == "bwd" else rnd
    return q, k, v, do


def _expected_codes(mask, d):
    """code[i, c] = sum_t M[i, c + d t] 2^t (forward: rows are queries)."""
    n = mask.shape[0]
    return sum(mask[:, t * d:(t + 1) * d].astype(np.int64) << t for t in range(n // d))


# p = 0.5 and below: byte thresholds t <= 128; 0.6 and 0.75: t = 154 and 192,
# the keep test's other branch (a byte is kept only with its top bit set)
@pytest.mark.parametrize("d,p", [(64, 0.1), (64, 0.5), (128, 0.25), (64, 0.75), (128, 0.6)])
def test_forward_mask_bit_exact(d, p):
    B, H, N = 2, 3, 4 * d
    q, k, v, do = _codes_inputs(B, H, N, d, "fwd")
    g = [t.cuda() for t in (q, k, v)]
    o, lse = fa.fa_fwd_dropout(*g, dropout_p=p, seed=SEED, offset=5, causal=False, scale=0.125)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    keep = dropout.keep_probability(p)
    o = o.float().cpu().double().numpy()
    for b in range(B):
        for h in range(H):
            mask = dropout.keep_mask(b * H + h, N, N, p, SEED, 5)
            got = np.rint(o[b, h] * N * keep).astype(np.int64)
            assert (got == _expected_codes(mask, d)).all(), (b, h)
    np.testing.assert_allclose(lse.cpu().numpy(), math.log(N), rtol=0, atol=1e-5)


# p = 0.5 and below: byte thresholds t <= 128; 0.6 and 0.75: t = 154 and 192,
# the keep test's other branch (a byte is kept only with its top bit set)
@pytest.mark.parametrize("d,p", [(64, 0.1), (64, 0.5), (128, 0.25), (64, 0.75), (128, 0.6)])
def test_backward_mask_bit_exact(d, p):
    B, H, N = 2, 3, 4 * d
    q, k, v, do = _codes_inputs(B, H, N, d, "bwd")
    g = [t.cuda() for t in (q, k, v, do)]
    o, lse = fa.fa_fwd_dropout(g[0], g[1], g[2], dropout_p=p, seed=SEED, offset=9, scale=0.125)
    dq, dk, dv = fa.fa_bwd_dropout(g[0], g[1], g[2], o, lse, g[3], dropout_p=p, seed=SEED, offset=9,
                                   scale=0.125)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    keep = dropout.keep_probability(p)
    dv = dv.float().cpu().double().numpy()
    for b in range(B):
        for h in range(H):
            mask = dropout.keep_mask(b * H + h, N, N, p, SEED, 9)
            # dV[j, c] = sum_t M[c + d t, j] 2^t / (N keep): rows of dV are keys
            got = np.rint(dv[b, h] * N * keep).astype(np.int64)
            assert (got == _expected_codes(mask.T, d)).all(), (b, h)


CASES = [
    (1, 2, 256, 64, True, 0.1),
    (2, 1, 200, 64, False, 0.3),
    (1, 1, 1, 64, True, 0.5),
    (1, 2, 333, 64, True, 0.2),
    (1, 2, 256, 128, True, 0.1),
    (2, 1, 300, 128, False, 0.25),
]


@pytest.mark.parametrize("B,H,N,d,causal,p", CASES)
def test_against_oracle(B, H, N, d, causal, p):
    x = si.make_small(B, H, N, d, seed=3000 + N + d, with_grad=True)
    scale = 1.0 / math.sqrt(d)
    g = {n: t.cuda() for n, t in x.items()}
    o, lse = fa.fa_fwd_dropout(g["q"], g["k"], g["v"], dropout_p=p, seed=SEED, offset=N,
                               causal=causal, scale=scale)
    dq, dk, dv = fa.fa_bwd_dropout(g["q"], g["k"], g["v"], o, lse, g["do"], dropout_p=p, seed=SEED,
                                   offset=N, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    o_ref, lse_ref = dropout.forward(x["q"], x["k"], x["v"], causal, scale, p, SEED, N)
    err = np.abs(o.float().cpu().double().numpy() - o_ref)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
    assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= 1e-3
    refs = dropout.backward(x["q"], x["k"], x["v"], o_ref, lse_ref, x["do"], causal, scale, p, SEED, N)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        gg = got.float().cpu().double().numpy()
        rel = float(np.abs(gg - ref).max() / max(np.abs(ref).max(), 1e-3))
        assert rel <= 5e-2, (name, rel)


def test_zero_probability_is_plain_attention():
    x = si.make_small(1, 2, 300, 64, seed=31, with_grad=True)
    g = {n: t.cuda() for n, t in x.items()}
    o0, l0 = fa.fa_fwd(g["q"], g["k"], g["v"], causal=True)
    o1, l1 = fa.fa_fwd_dropout(g["q"], g["k"], g["v"], dropout_p=0.0, seed=1, causal=True)
    d0 = fa.fa_bwd(g["q"], g["k"], g["v"], o0, l0, g["do"], causal=True)
    d1 = fa.fa_bwd_dropout(g["q"], g["k"], g["v"], o1, l1, g["do"], dropout_p=0.0, seed=1, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    for a, b in zip(d0, d1):
        assert torch.equal(a, b)


def test_offset_changes_the_mask_and_repeats_are_identical():
    x = si.make_small(1, 1, 256, 64, seed=32, with_grad=False)
    g = {n: t.cuda() for n, t in x.items()}
    a, _ = fa.fa_fwd_dropout(g["q"], g["k"], g["v"], dropout_p=0.5, seed=7, offset=1)
    b, _ = fa.fa_fwd_dropout(g["q"], g["k"], g["v"], dropout_p=0.5, seed=7, offset=1)
    c, _ = fa.fa_fwd_dropout(g["q"], g["k"], g["v"], dropout_p=0.5, seed=7, offset=2)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert not torch.equal(a, c)


def test_fwdbwd_workload_full_size():
    """The forward+backward workload at full size (B=8, H=12, N=2048, d=64, causal) with p = 0.1,
    the configuration the bench's dropout leg times: every head against the oracle, head by head,
    and finite outputs and sum_j dK_j = 0 (row sums of dS vanish with dropout too, because
    D_i = sum_j P_ij dP_ij)."""
    w = si.workload("causal_fwdbwd_b8h12_n2048_d64")
    x = si.make_inputs(w)
    g = {n: t.cuda() for n, t in x.items()}
    p, seed, offset = 0.1, 2024, 1
    o, lse = fa.fa_fwd_dropout(g["q"], g["k"], g["v"], p, seed, offset, causal=True, scale=w.scale)
    dq, dk, dv = fa.fa_bwd_dropout(g["q"], g["k"], g["v"], o, lse, g["do"], p, seed, offset, causal=True,
                                   scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    o_ref, lse_ref = dropout.forward(x["q"], x["k"], x["v"], True, w.scale, p, seed, offset)
    refs = dropout.backward(x["q"], x["k"], x["v"], o_ref, lse_ref, x["do"], True, w.scale, p, seed, offset)
    o_np, lse_np = o.float().cpu().double().numpy(), lse.cpu().double().numpy()
    for b, h in heads:
        err = np.abs(o_np[b, h] - o_ref[b, h])
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, ((b, h), err.max(), err.mean())
        assert np.abs(lse_np[b, h] - lse_ref[b, h]).max() <= 1e-3
        for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
            gg = got[b, h].float().cpu().double().numpy()
            rel = float(np.abs(gg - ref[b, h]).max() / max(np.abs(ref[b, h]).max(), 1e-3))
            assert rel <= 5e-2, ((b, h), name, rel)
    for t in (o, dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    dkf = dk.float()
    assert float(dkf.sum(dim=2).abs().max()) <= 2e-2 * float(dkf.abs().sum(dim=2).max())
