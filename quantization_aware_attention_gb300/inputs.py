"""Seeded synthetic inputs for QAT attention (shared by the tests, the oracle checks
and the benchmark).  This module holds no attention or quantization arithmetic: it
draws normal samples and rounds them to bf16 bit patterns.

Workloads (all bf16 [B, H, N, D], standard normal unless stated):
  c1  B1 H2  N256           D128  non-causal          quant tile 64, several tiles
  c2  B2 H4  N8             D64   non-causal          shorter than one tile (padding)
  c3  B1 H24 N4608          D128  non-causal          K += mu (per channel, mu ~ N(0, 2^2))
  c4  B1 H40 N32768         D128  non-causal          long video-DiT self-attention
  c5a B4 H32 N8192          D128  causal              LM-style
  c5b B1 H40 Nq16384 Nkv512 D128  non-causal          cross-attention
sm_scale = 1 / sqrt(D).  Seeds: q = 1000 * idx, k = +1, v = +2, dO = +3, mu = +4,
with idx 1..6 in the order above.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    idx: int
    B: int
    H: int
    Nq: int
    Nkv: int
    D: int
    causal: bool = False
    k_offset_sigma: float = 0.0

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def pairs(self) -> int:
        """Unmasked (i, j) score entries summed over all heads."""
        per_head = self.Nq * (self.Nq + 1) // 2 if self.causal else self.Nq * self.Nkv
        return self.B * self.H * per_head


WORKLOADS = {
    "c1": Workload("c1", 1, 1, 2, 256, 256, 128),
    "c2": Workload("c2", 2, 2, 4, 8, 8, 64),
    "c3": Workload("c3", 3, 1, 24, 4608, 4608, 128, k_offset_sigma=2.0),
    "c4": Workload("c4", 4, 1, 40, 32768, 32768, 128),
    "c5a": Workload("c5a", 5, 4, 32, 8192, 8192, 128, causal=True),
    "c5b": Workload("c5b", 6, 1, 40, 16384, 512, 128),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 samples to bf16 (nearest, ties to even) and return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def normal_bf16(seed: int, shape) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return f32_to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def make_inputs(w: Workload, with_do: bool = True) -> dict:
    """bf16 bit patterns (uint16) for q, k, v (and dO) of workload ``w``."""
    base = 1000 * w.idx
    q = normal_bf16(base + 0, (w.B, w.H, w.Nq, w.D))
    if w.k_offset_sigma:
        rng = np.random.default_rng(base + 1)
        k32 = rng.standard_normal(size=(w.B, w.H, w.Nkv, w.D), dtype=np.float32)
        mu = (np.random.default_rng(base + 4).standard_normal(size=(w.D,), dtype=np.float32)
              * np.float32(w.k_offset_sigma))
        k = f32_to_bf16_bits(k32 + mu)
    else:
        k = normal_bf16(base + 1, (w.B, w.H, w.Nkv, w.D))
    v = normal_bf16(base + 2, (w.B, w.H, w.Nkv, w.D))
    out = {"q": q, "k": k, "v": v}
    if with_do:
        out["do"] = normal_bf16(base + 3, (w.B, w.H, w.Nq, w.D))
    return out


def custom_inputs(seed: int, B: int, H: int, Nq: int, Nkv: int, D: int) -> dict:
    """Standard-normal bf16 q, k, v, dO of an arbitrary shape (edge-case tests)."""
    return {
        "q": normal_bf16(seed + 0, (B, H, Nq, D)),
        "k": normal_bf16(seed + 1, (B, H, Nkv, D)),
        "v": normal_bf16(seed + 2, (B, H, Nkv, D)),
        "do": normal_bf16(seed + 3, (B, H, Nq, D)),
    }
