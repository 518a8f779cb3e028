"""Philox4x32 outputs from Triton's own implementation, for the oracle's pin.

Run as a script with ``TRITON_INTERPRET=1`` set, so that Triton executes the
kernel on the CPU through its interpreter (no GPU involved). Reads a JSON
object ``{"ctr": [[c0, c1, c2, c3], ...], "key": [[k0, k1], ...],
"rounds": R}`` from standard input and writes the list of output words
``[[x0, x1, x2, x3], ...]`` to standard output.

Triton ships a Philox4x32 of its own (``triton.language.philox_impl``),
written independently of this repository; comparing the oracle's generator
with it checks the multipliers, the Weyl increments, the word order of each
round and the key schedule at once.
"""

import json
import os
import sys

import numpy as np


def main():
    if os.environ.get("TRITON_INTERPRET") != "1":
        raise SystemExit("set TRITON_INTERPRET=1 (the kernel runs on the CPU interpreter)")
    import torch
    import triton
    import triton.language as tl

    req = json.load(sys.stdin)
    ctr = np.asarray(req["ctr"], dtype=np.uint64).astype(np.uint32)
    key = np.asarray(req["key"], dtype=np.uint64).astype(np.uint32)
    rounds = int(req.get("rounds", 10))
    n = ctr.shape[0]

    @triton.jit
    def kernel(c_ptr, k_ptr, out_ptr, n, ROUNDS: tl.constexpr, BLOCK: tl.constexpr):
        i = tl.program_id(0) * BLOCK + tl.arange(0, BLOCK)
        m = i < n
        c0 = tl.load(c_ptr + 4 * i + 0, mask=m)
        c1 = tl.load(c_ptr + 4 * i + 1, mask=m)
        c2 = tl.load(c_ptr + 4 * i + 2, mask=m)
        c3 = tl.load(c_ptr + 4 * i + 3, mask=m)
        k0 = tl.load(k_ptr + 2 * i + 0, mask=m)
        k1 = tl.load(k_ptr + 2 * i + 1, mask=m)
        x0, x1, x2, x3 = tl.philox_impl(c0, c1, c2, c3, k0, k1, ROUNDS)
        tl.store(out_ptr + 4 * i + 0, x0, mask=m)
        tl.store(out_ptr + 4 * i + 1, x1, mask=m)
        tl.store(out_ptr + 4 * i + 2, x2, mask=m)
        tl.store(out_ptr + 4 * i + 3, x3, mask=m)

    as_u32 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).view(torch.uint32)
    out = torch.zeros((n, 4), dtype=torch.uint32)
    block = 64
    kernel[((n + block - 1) // block,)](as_u32(ctr), as_u32(key), out, n, ROUNDS=rounds, BLOCK=block)
    words = out.view(torch.int32).numpy().view(np.uint32)
    json.dump([[int(w) for w in row] for row in words], sys.stdout)


if __name__ == "__main__":
    main()
