"""Pins of the oracle's Philox4x32-10 generator (CPU only).

The dropout mask is drawn from Philox4x32-10 (Salmon, Moraes, Dror and Shaw,
"Parallel random numbers: as easy as 1, 2, 3", SC 2011). Statistical checks
(kept fraction, uniformity, avalanche) cannot tell that generator from a
near miss, so the generator itself is pinned here, by two things that do not
come from the oracle:

* Triton's independent Philox4x32 (``triton.language.philox_impl``), run on
  the CPU through Triton's interpreter in a child process: the oracle must
  give the same four words for every counter and key tried, edge values
  (all-zero and all-ones words) included, at 10 rounds and at 1, 2 and 7
  rounds (so that a mistake in the key schedule of a single round shows);
* the closed forms of the two Weyl key increments: the first 32 fractional
  bits of the golden ratio, floor(2^32 (sqrt(5) - 1) / 2), and of sqrt(3),
  floor(2^32 (sqrt(3) - 1)).

Planted mistakes (swapped multipliers, a wrong increment, the high and low
product words exchanged, the key bumped before the first round, the words
of a round permuted) must each fail the comparison.
"""

import json
import math
import os
import subprocess
import sys

import numpy as np
import pytest

from oracle import dropout

HERE = os.path.dirname(os.path.abspath(__file__))
M32 = 0xFFFFFFFF


def _cases():
    """Counters and keys: edge words, single set bits, then random ones."""
    rng = np.random.default_rng(20111112)
    ctr, key = [], []
    edge = [0, 1, 0x80000000, M32]
    for a in edge:
        for b in edge:
            ctr.append([a, b, a ^ M32, b])
            key.append([b, a])
    for bit in range(0, 32, 5):
        ctr.append([1 << bit, 0, 0, 0])
        key.append([0, 1 << bit])
        ctr.append([0, 0, 1 << bit, 1 << (31 - bit)])
        key.append([1 << bit, 0])
    r = rng.integers(0, 2**32, size=(200, 6), dtype=np.uint64)
    ctr += r[:, :4].tolist()
    key += r[:, 4:].tolist()
    return np.asarray(ctr, dtype=np.uint64), np.asarray(key, dtype=np.uint64)


@pytest.fixture(scope="module")
def triton_words():
    """{rounds: uint32 [n, 4]} from Triton's Philox on the cases above."""
    pytest.importorskip("triton")
    ctr, key = _cases()
    out = {}
    env = dict(os.environ, TRITON_INTERPRET="1", CUDA_VISIBLE_DEVICES="")
    for rounds in (1, 2, 7, 10):
        req = json.dumps({"ctr": ctr.tolist(), "key": key.tolist(), "rounds": rounds})
        res = subprocess.run([sys.executable, os.path.join(HERE, "_philox_triton.py")], input=req,
                             capture_output=True, text=True, env=env, timeout=600)
        if res.returncode != 0:
            pytest.skip(f"Triton interpreter unavailable: {res.stderr.strip()[-300:]}")
        out[rounds] = np.asarray(json.loads(res.stdout), dtype=np.uint64).astype(np.uint32)
    return out


def _oracle_words(gen, rounds):
    ctr, key = _cases()
    rows = []
    for c, k in zip(ctr, key):
        w = gen(c[0], c[1], c[2], c[3], int(k[0]), int(k[1]), rounds)
        rows.append([int(x) for x in w])
    return np.asarray(rows, dtype=np.uint64).astype(np.uint32)


def check_against_triton(gen, triton_words):
    for rounds, ref in triton_words.items():
        got = _oracle_words(gen, rounds)
        bad = np.nonzero((got != ref).any(axis=1))[0]
        assert bad.size == 0, f"{rounds} rounds: {bad.size} of {len(ref)} cases differ (first {bad[:5]})"


def test_oracle_generator_matches_triton(triton_words):
    check_against_triton(dropout.philox4x32, triton_words)


def test_weyl_increments_are_the_published_irrationals():
    # first 32 fractional bits of the golden ratio (sqrt(5) - 1) / 2 ...
    golden = (math.isqrt(5 << 64) - (1 << 32)) // 2
    # ... and of sqrt(3) - 1
    root3 = math.isqrt(3 << 64) - (1 << 32)
    assert int(dropout._W0) == golden == 0x9E3779B9
    assert int(dropout._W1) == root3 == 0xBB67AE85


def test_keep_bytes_use_the_generator_words():
    # byte (j & 3) of word (i & 3) of the call for key group j >> 2, query group i >> 2
    seed, offset, bh = 0x0123456789ABCDEF, 0x55, 7
    b = dropout.keep_bytes(bh, 8, 8, seed, offset)
    for qg in range(2):
        for kg in range(2):
            w = dropout.philox4x32(kg, qg, bh, offset, seed & M32, seed >> 32)
            for qi in range(4):
                for kj in range(4):
                    assert b[4 * qg + qi, 4 * kg + kj] == (int(w[qi]) >> (8 * kj)) & 0xFF


# --------------------------------------------------------------------------
# Planted mistakes: each near miss of the generator must fail the pin.
# --------------------------------------------------------------------------

def _variant(m0=0xD2511F53, m1=0xCD9E8D57, w0=0x9E3779B9, w1=0xBB67AE85, swap_hilo=False,
             bump_first=False, permute=False):
    """The Philox round function with one knob turned (a restatement made for
    the planted-mistake tests only)."""

    def gen(c0, c1, c2, c3, k0, k1, rounds=10):
        c = [int(c0) & M32, int(c1) & M32, int(c2) & M32, int(c3) & M32]
        k0, k1 = k0 & M32, k1 & M32
        for r in range(rounds):
            if r > 0 or bump_first:
                k0, k1 = (k0 + w0) & M32, (k1 + w1) & M32
            p0, p1 = c[0] * m0, c[2] * m1
            hi0, lo0 = p0 >> 32, p0 & M32
            hi1, lo1 = p1 >> 32, p1 & M32
            if swap_hilo:
                hi0, lo0, hi1, lo1 = lo0, hi0, lo1, hi1
            c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
            if permute:
                c = [c[2], c[1], c[0], c[3]]
        return c

    return gen


def test_restated_variant_without_a_mistake_passes(triton_words):
    check_against_triton(_variant(), triton_words)


@pytest.mark.parametrize("mistake", [
    {"m0": 0xCD9E8D57, "m1": 0xD2511F53},   # multipliers swapped
    {"w0": 0x9E3779B7},                      # golden-ratio increment off by two
    {"w1": 0x9E3779B9},                      # both keys bumped by the same increment
    {"swap_hilo": True},                     # high and low product words exchanged
    {"bump_first": True},                    # key bumped before the first round
    {"permute": True},                       # output words of a round in the wrong order
], ids=["multipliers-swapped", "weyl0-off", "weyl1-wrong", "hi-lo-swapped", "key-bumped-early",
        "words-permuted"])
def test_planted_mistake_is_caught(mistake, triton_words):
    with pytest.raises(AssertionError):
        check_against_triton(_variant(**mistake), triton_words)
