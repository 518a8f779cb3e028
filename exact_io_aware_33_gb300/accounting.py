"""Algorithmic work and traffic of exact attention (host-side bookkeeping).

These counts are what the throughput and roofline figures divide by; they
describe the method, not what any kernel happens to do.

* Forward FLOPs: 4 B H N^2 d (two N x N x d contractions, QK^T and PV, at
  2 FLOPs per multiply-add), halved under a causal mask.
* Backward FLOPs: 2.5 x the forward (five contractions instead of two).
* Forward bytes: Q, K, V read and O written once in bf16, LSE written in
  fp32: 8 B H N d + 4 B H N.
* Backward bytes: Q, K, V, O, dO read and dQ, dK, dV written in bf16, LSE
  and D in fp32: 16 B H N d + 8 B H N.

``transfer_ledger`` restates the element-transfer count of the explorer of
"Flash Attention: IO-Aware Exact Attention", section "Loop order changes
which data is reloaded": under the query-resident schedule every query
block reads all of K and V once, and the dense path additionally writes and
reads the N x N scores and probabilities.
"""

from __future__ import annotations


def flops_fwd(B: int, H: int, N: int, d: int, causal: bool) -> float:
    f = 4.0 * B * H * N * N * d
    return f * 0.5 if causal else f


def flops_bwd(B: int, H: int, N: int, d: int, causal: bool) -> float:
    return 2.5 * flops_fwd(B, H, N, d, causal)


def bytes_fwd(B: int, H: int, N: int, d: int) -> int:
    return 8 * B * H * N * d + 4 * B * H * N


def bytes_bwd(B: int, H: int, N: int, d: int) -> int:
    return 16 * B * H * N * d + 8 * B * H * N


def transfer_ledger(N: int, d: int, d_v: int, query_block: int) -> dict:
    """Element transfers of one head's forward, tiled versus dense."""
    blocks = -(-N // query_block)
    reads = {"Q": N * d, "K": blocks * N * d, "V": blocks * N * d_v}
    writes = {"O": N * d_v}
    tiled = sum(reads.values()) + sum(writes.values())
    dense = tiled + 4 * N * N
    return {"reads": reads, "writes": writes, "tiled_total": tiled, "dense_total": dense}
