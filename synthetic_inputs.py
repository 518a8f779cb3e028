"""Seeded synthetic workloads for exact attention.

This module is shared by the CPU oracle (``oracle/``), the CUDA path's tests
and ``bench.py``. It only draws and shapes random numbers; it holds none of
the attention arithmetic, so neither side can lean on the other through it.

Every tensor is drawn on the CPU from ``torch.Generator().manual_seed(seed)``
as float32 ``randn`` in the fixed order q, k, v, dO, then rounded to bfloat16
(round-to-nearest-even). Where a workload scales a tensor (the ragged
workload's keys), the scaling happens in float32 before the rounding, so the
stored bfloat16 values are what both sides read.

Layout: ``[B, H, N, d]`` contiguous row-major, the (batch, heads, sequence,
head size) order of the dense PyTorch attention block shown in
"FlashAttention -- the same attention, made memory-aware", section 00.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = ["Workload", "WORKLOADS", "workload", "make_inputs", "make_small"]


@dataclass(frozen=True)
class Workload:
    """One attention problem: sizes, mask, scale and the seed of its inputs."""

    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    backward: bool = False
    k_mult: float = 1.0
    seed: int = 0
    note: str = ""
    scale: float = field(default=float("nan"))

    def __post_init__(self):
        if math.isnan(self.scale):
            object.__setattr__(self, "scale", 1.0 / math.sqrt(self.d))

    @property
    def heads(self) -> int:
        return self.B * self.H

    def as_dict(self) -> dict:
        return {
            "workload": self.name,
            "B": self.B,
            "H": self.H,
            "N": self.N,
            "d": self.d,
            "causal": self.causal,
            "backward": self.backward,
            "scale": self.scale,
            "k_mult": self.k_mult,
            "seed": self.seed,
        }


# The five workloads the attention library is checked and measured on. The
# second mirrors GPT-2-small attention (12 heads of size 64, 1024 tokens);
# none of them needs a dataset or trained weights.
WORKLOADS = [
    Workload("single_head_n256_d64", 1, 1, 256, 64, False, seed=1001,
             note="one head, non-causal, forward only"),
    Workload("gpt2s_causal_b8h12_n1024_d64", 8, 12, 1024, 64, True, seed=1002,
             note="GPT-2-small shaped causal forward"),
    Workload("ragged_b4h32_n1000_d128_k3", 4, 32, 1000, 128, False, k_mult=3.0, seed=1003,
             note="N not a multiple of the tile; keys scaled x3 so row maxima move"),
    Workload("long_causal_b1h16_n8192_d128", 1, 16, 8192, 128, True, seed=1004,
             note="long-sequence causal forward; memory linear in N"),
    Workload("causal_fwdbwd_b8h12_n2048_d64", 8, 12, 2048, 64, True, backward=True, seed=1005,
             note="causal forward + backward by recomputation"),
]


def workload(name_or_index) -> Workload:
    if isinstance(name_or_index, int):
        return WORKLOADS[name_or_index]
    for w in WORKLOADS:
        if w.name == name_or_index:
            return w
    raise KeyError(name_or_index)


def make_inputs(w: Workload, with_grad: bool | None = None) -> dict:
    """Return bf16 CPU tensors q, k, v (and dO when the workload has a backward).

    Draw order is always q, k, v, dO so that a forward-only and a
    forward+backward draw of the same seed agree on q, k, v.
    """
    if with_grad is None:
        with_grad = w.backward
    return make_small(w.B, w.H, w.N, w.d, seed=w.seed, k_mult=w.k_mult, with_grad=with_grad)


def make_small(B: int, H: int, N: int, d: int, seed: int, k_mult: float = 1.0,
               with_grad: bool = True, dtype=torch.bfloat16) -> dict:
    """Draw iid N(0,1) q, k, v, dO of shape [B,H,N,d] and round them to ``dtype``."""
    g = torch.Generator().manual_seed(seed)
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    out = {}
    if with_grad:
        do = torch.randn(shape, generator=g, dtype=torch.float32)
        out["do"] = do.to(dtype).contiguous()
    if k_mult != 1.0:
        k = k * k_mult
    out["q"] = q.to(dtype).contiguous()
    out["k"] = k.to(dtype).contiguous()
    out["v"] = v.to(dtype).contiguous()
    return out
