"""CPU oracle for exact scaled-dot-product attention -- TEST INFRASTRUCTURE.

This package is a plain, slow, float64 restatement of what the attention
library computes. It exists only to check the CUDA path: the tests, the
``smoke()`` check and the timed CPU baseline of ``bench.py`` may import it;
the library itself never does, and the oracle imports nothing from the
library. The two share no code; the only common module is the seeded input
generator, which holds no attention arithmetic.

Modules
-------
dense
    The definition written out: S = scale * Q K^T, optional causal mask,
    row softmax, O = P V, LSE = m + ln(l); and the gradients of
    L = sum(O * dO) with respect to Q, K, V.
tiled
    The query-block-outer, key-block-inner online-softmax recurrence in the
    order the pages give it, with the causal mask and ragged tail tiles.
finite_diff
    Central finite differences of L = sum(O * dO), for pinning the backward.
general
    The dense definition with Nq queries over Nk keys (causal queries are the
    last Nq positions), an optional sliding window and key-range restriction.
merge
    The page's rule for merging partial softmax states, applied to the parts
    of a split key range.
dropout
    Dropout on the probabilities with a keep mask drawn from Philox4x32-10,
    and the forward and backward for a given mask.

Pins (what fixes each function other than itself) live in
``tests/test_oracle_pins.py``, ``tests/test_oracle_general.py``,
``tests/test_oracle_dropout.py`` and ``tests/test_oracle_philox.py``; each
module's docstring names its pins.
No function here is "parity unpinned".

Sources cited (title of the page, then its section):
  * "Flash Attention: IO-Aware Exact Attention" (abhik.ai)
  * "FlashAttention -- the same attention, made memory-aware" (plasmient.com)
  * "FlashAttention" (Road to Intelligence, Chapter 11)
"""

from . import dense, tiled, finite_diff, general, merge, dropout  # noqa: F401

__all__ = ["dense", "tiled", "finite_diff", "general", "merge", "dropout"]
