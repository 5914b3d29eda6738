"""Seeded synthetic workloads: shapes of the five attention problems and their inputs.

This module holds no attention arithmetic.  It only says which problem sizes are
run and how the packed ``qkv[B,S,H,3,D]`` bf16 inputs are drawn, so that the CUDA
path, the oracle, the tests and the benchmark all see the same bytes.

Shapes (head count, head dim, rotary dims, 2048-token context) follow the
GPT-NeoX family: the GPT-NeoX-20B numbers (64 heads x 96 dims, 24 rotary dims)
are printed in the FasterTransformer guide's "模型配置（config.ini）" section and
the 2048-token window in the GPT-NeoX-20B release article.

Input recipe: ``torch.Generator().manual_seed(seed)``, ``torch.randn`` in fp32 of
shape ``[B,S,H,3,D]``, the K slot multiplied by ``k_scale`` (3 for the
long-context case, to sharpen the softmax), then cast to bf16 (round to nearest
even).  Scaling happens before the cast so the stored input is what both sides
read.  ``seed = 1000 + index`` (index 1..5).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    B: int
    H: int
    S: int
    D: int
    rotary_dim: int
    rotary_base: float = 10000.0
    k_scale: float = 1.0

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def flops(self) -> float:
        """Causal attention forward FLOPs, 2*B*H*S^2*D (QK^T and PV over the causal half)."""
        return 2.0 * self.B * self.H * self.S * self.S * self.D

    @property
    def qkv_shape(self):
        return (self.B, self.S, self.H, 3, self.D)

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "S": self.S, "D": self.D,
                "rotary_dim": self.rotary_dim, "rotary_base": self.rotary_base, "k_scale": self.k_scale,
                "seed": self.seed}


WORKLOADS = {
    "tiny": Workload("tiny", 1, B=1, H=2, S=128, D=64, rotary_dim=16),
    "pythia160m": Workload("pythia160m", 2, B=8, H=12, S=2048, D=64, rotary_dim=16),
    "pythia1.4b": Workload("pythia1.4b", 3, B=4, H=16, S=2048, D=128, rotary_dim=32),
    "neox20b": Workload("neox20b", 4, B=2, H=64, S=2048, D=96, rotary_dim=24),
    "long16k": Workload("long16k", 5, B=1, H=32, S=16384, D=128, rotary_dim=128, k_scale=3.0),
}


def make_qkv(B: int, S: int, H: int, D: int, seed: int, k_scale: float = 1.0) -> torch.Tensor:
    """Packed ``qkv[B,S,H,3,D]`` bf16 on the CPU, N(0,1) with the K slot scaled by ``k_scale``."""
    g = torch.Generator().manual_seed(int(seed))
    x = torch.randn((B, S, H, 3, D), generator=g, dtype=torch.float32)
    if k_scale != 1.0:
        x[:, :, :, 1, :] *= k_scale
    return x.to(torch.bfloat16)


def workload_qkv(w: Workload) -> torch.Tensor:
    return make_qkv(w.B, w.S, w.H, w.D, w.seed, w.k_scale)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw 16-bit patterns of a CPU bf16 tensor, as numpy.uint16 (no copy of values)."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_rows(w: Workload, n: int = 256, extra_edges: bool = True) -> np.ndarray:
    """Seeded (b, h, i) triples: ``n`` distinct uniform draws (numpy default_rng(seed+1)),
    plus fixed edge rows {0, 1, 127, 128, S-1} of head (0, 0) that fall inside S."""
    rng = np.random.default_rng(w.seed + 1)
    total = w.B * w.H * w.S
    flat = rng.choice(total, size=min(n, total), replace=False)
    b = flat // (w.H * w.S)
    h = (flat // w.S) % w.H
    i = flat % w.S
    rows = np.stack([b, h, i], axis=1).astype(np.int64)
    if extra_edges:
        edges = sorted({e for e in (0, 1, 127, 128, w.S - 1) if 0 <= e < w.S})
        rows = np.concatenate([rows, np.array([[0, 0, e] for e in edges], dtype=np.int64)], axis=0)
    return rows
