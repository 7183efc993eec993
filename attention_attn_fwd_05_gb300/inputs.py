"""Seeded synthetic inputs for attention forward.

This module only draws random numbers and names workloads; it holds none of
the method's arithmetic.  It is the one module that both the CUDA path's
tests/bench and the CPU oracle's callers use, so that both sides see the same
values.

Recipe: a CPU ``torch.Generator`` seeded with the workload's seed draws Q,
then K, then V, each a float32 ``[B, H, N, d]`` tensor.  ``normal`` is
``randn``; ``stress`` draws Q and K as ``4 * randn`` (variance 16, so logits
have a standard deviation near 16) and V as ``2 * rand - 1`` (uniform on
[-1, 1)).  For bf16 workloads the float32 draws are rounded to bf16
(round-to-nearest-even) on the host; the oracle then reads those bf16 values
widened back to float32, i.e. exactly what the GPU sees.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    """One attention-forward problem: shapes, dtype, mask and input recipe."""
    name: str
    dtype: str          # "f32" or "bf16": input, output and MMA operand type
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    dist: str = "normal"  # "normal" or "stress"

    @property
    def scale(self) -> float:
        """1/sqrt(d), rounded to float32 (the value both sides use)."""
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32))

    @property
    def flops(self) -> float:
        """4*B*H*N^2*d, halved with the causal mask (nominal count)."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def io_bytes(self) -> int:
        """Algorithmic HBM bytes: read Q, K, V once; write O once and LSE (fp32)."""
        n = self.B * self.H * self.N * self.d
        return 4 * n * self.elem_bytes + self.B * self.H * self.N * 4


# The problem shapes the method is measured and checked on.
WORKLOADS = {
    w.name: w for w in [
        Workload("f32_B1_H1_N128_d64", "f32", 1, 1, 128, 64, False, 0),
        Workload("f32_B1_H8_N1024_d64", "f32", 1, 8, 1024, 64, False, 1),
        Workload("bf16_B1_H8_N1024_d64", "bf16", 1, 8, 1024, 64, False, 1),
        Workload("bf16_B4_H16_N2048_d128", "bf16", 4, 16, 2048, 128, False, 2),
        Workload("bf16_B4_H16_N2048_d128_causal", "bf16", 4, 16, 2048, 128, True, 2),
        Workload("bf16_B1_H32_N16384_d128_causal", "bf16", 1, 32, 16384, 128, True, 3),
        Workload("bf16_B2_H16_N4000_d128_causal_stress", "bf16", 2, 16, 4000, 128, True, 4,
                 "stress"),
        # The long causal sequence again at head dimension 64.
        Workload("bf16_B1_H32_N16384_d64_causal", "bf16", 1, 32, 16384, 64, True, 5),
    ]
}


def torch_dtype(dtype: str) -> torch.dtype:
    if dtype == "f32":
        return torch.float32
    if dtype == "bf16":
        return torch.bfloat16
    raise ValueError(f"unknown dtype {dtype!r}")


def make_qkv(B: int, H: int, N: int, d: int, seed: int, dtype: str = "bf16",
             dist: str = "normal"):
    """Draw (Q, K, V) on the CPU in the workload's dtype, per the module recipe."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    shape = (B, H, N, d)
    if dist == "normal":
        q = torch.randn(shape, generator=g, dtype=torch.float32)
        k = torch.randn(shape, generator=g, dtype=torch.float32)
        v = torch.randn(shape, generator=g, dtype=torch.float32)
    elif dist == "stress":
        q = 4.0 * torch.randn(shape, generator=g, dtype=torch.float32)
        k = 4.0 * torch.randn(shape, generator=g, dtype=torch.float32)
        v = 2.0 * torch.rand(shape, generator=g, dtype=torch.float32) - 1.0
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    t = torch_dtype(dtype)
    return q.to(t), k.to(t), v.to(t)


def make_workload_inputs(w: Workload):
    return make_qkv(w.B, w.H, w.N, w.d, w.seed, w.dtype, w.dist)


def make_rows(rows: int, width: int, seed: int, spread: float = 1.0):
    """A float32 [rows, width] matrix of ``spread * randn`` for the row softmax."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    return spread * torch.randn((rows, width), generator=g, dtype=torch.float32)
