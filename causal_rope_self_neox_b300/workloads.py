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


# ------------------------------------------------------------------ decode ----
# Incremental decode: one new token per sequence against a cache of earlier tokens.
# The cache holds the projections as they came (keys not rotated), head-major
# [B, H, Smax, D]; the new token's packed projection is [B, H, 3, D].

@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    index: int
    B: int
    H: int
    Smax: int
    D: int
    rotary_dim: int
    pos: int  # tokens already cached in every sequence (the new token's position)
    rotary_base: float = 10000.0

    @property
    def seed(self) -> int:
        return 2000 + self.index

    @property
    def cache_bytes_read(self) -> int:
        """K and V cache rows read per step (bf16): 2 * B * H * pos * D * 2."""
        return 4 * self.B * self.H * self.pos * self.D

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "H": self.H, "Smax": self.Smax, "D": self.D,
                "rotary_dim": self.rotary_dim, "rotary_base": self.rotary_base, "pos": self.pos,
                "seed": self.seed}


# serving-style batches at the end of a 2048-token context (GPT-NeoX family shapes)
DECODE_WORKLOADS = {
    "neox20b-decode": DecodeWorkload("neox20b-decode", 1, B=16, H=64, Smax=2048, D=96, rotary_dim=24, pos=2047),
    "pythia1.4b-decode": DecodeWorkload("pythia1.4b-decode", 2, B=32, H=16, Smax=2048, D=128, rotary_dim=32,
                                        pos=2047),
    "pythia160m-decode": DecodeWorkload("pythia160m-decode", 3, B=64, H=12, Smax=2048, D=64, rotary_dim=16,
                                        pos=2047),
}


def make_decode_inputs(B: int, H: int, Smax: int, D: int, seed: int):
    """(qkv_new [B,H,3,D], k_cache [B,H,Smax,D], v_cache [B,H,Smax,D]) bf16 on the CPU, N(0,1)."""
    g = torch.Generator().manual_seed(int(seed))
    qkv_new = torch.randn((B, H, 3, D), generator=g, dtype=torch.float32).to(torch.bfloat16)
    k_cache = torch.randn((B, H, Smax, D), generator=g, dtype=torch.float32).to(torch.bfloat16)
    v_cache = torch.randn((B, H, Smax, D), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return qkv_new, k_cache, v_cache


def decode_from_sequence(qkv: torch.Tensor, pos, Smax: int):
    """Split a prefill input qkv[B,S,H,3,D] into decode inputs: for sequence b the cache gets
    tokens 0..pos[b]-1 (rows >= pos[b] filled with a sentinel pattern that must never be read)
    and the new token is token pos[b].  Pure data movement."""
    B, S, H, _, D = qkv.shape
    new = torch.empty((B, H, 3, D), dtype=qkv.dtype)
    kc = torch.full((B, H, Smax, D), 12345.0, dtype=qkv.dtype)
    vc = torch.full((B, H, Smax, D), -12345.0, dtype=qkv.dtype)
    for b in range(B):
        p = int(pos[b])
        new[b] = qkv[b, p]
        kc[b, :, :p] = qkv[b, :p, :, 1].permute(1, 0, 2)
        vc[b, :, :p] = qkv[b, :p, :, 2].permute(1, 0, 2)
    return new, kc, vc


# ------------------------------------------------------- qkv projection ----
# The query_key_value projection that feeds the attention: token rows x[B*S, hidden] (the
# layer-normed hidden states), weight w[hidden, H, 3, D] (HuggingFace layout) and bias[3*H*D].
# hidden = H * D for the GPT-NeoX family (6144 = 64 x 96 for the 20B model).
# Recipe: one torch.Generator seeded with ``seed``; x ~ N(0, 1); w ~ N(0, 1) / sqrt(hidden)
# (so the projections are about unit-normal, the scale of the attention inputs above);
# bias ~ N(0, 0.5^2); each drawn in fp32 and cast to bf16 (round to nearest even).

def make_proj_inputs(B: int, S: int, hidden: int, H: int, D: int, seed: int, with_bias: bool = True):
    """``(x[B*S, hidden], w[hidden, 3*H*D], bias[3*H*D] or None)`` bf16 on the CPU."""
    g = torch.Generator().manual_seed(int(seed))
    N = 3 * H * D
    x = torch.randn((B * S, hidden), generator=g, dtype=torch.float32).to(torch.bfloat16)
    w = (torch.randn((hidden, N), generator=g, dtype=torch.float32) / float(np.sqrt(hidden))).to(torch.bfloat16)
    bias = (torch.randn((N,), generator=g, dtype=torch.float32) * 0.5).to(torch.bfloat16) if with_bias else None
    return x, w, bias


def proj_inputs(w: Workload, with_bias: bool = True):
    """The projection inputs of an attention workload: hidden = H * D, seed 3000 + index."""
    return make_proj_inputs(w.B, w.S, w.H * w.D, w.H, w.D, 3000 + w.index, with_bias)
