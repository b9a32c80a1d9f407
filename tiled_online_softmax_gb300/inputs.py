"""Seeded synthetic inputs for the attention forward pass.

This module only draws numbers and rounds them into the 16-bit storage types. It holds none of
the attention arithmetic and imports nothing else from this package, so both the CUDA path and
the CPU oracle can be fed from it without sharing code.

Recipe: Q, K and V are drawn i.i.d. normal in float32 from three independent NumPy PCG64
streams spawned from one seed, multiplied by their standard deviation, then rounded to the
nearest 16-bit value (ties to even): fp16 through NumPy's float16 cast, bf16 by rounding the
float32 bit pattern. The values are returned as raw 16-bit patterns, which the GPU reads as is
and the oracle widens exactly to float64.

Workloads are the ones attention kernels are measured on: a single head, a ragged multi-head
case, causal prefill, a large-magnitude case where the row maximum keeps moving, a long causal
context, and the headline shape (one batch, 32 heads, 4096 tokens, head dim 128).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np

F16, BF16 = 0, 1  # the fa_dtype codes of the C interface
DTYPE_CODES = {"f16": F16, "bf16": BF16}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    D: int
    dtype: str  # "f16" or "bf16"
    causal: bool
    seed: int
    sigma_q: float = 1.0
    sigma_k: float = 1.0
    sigma_v: float = 1.0
    scale: float = field(default=float("nan"))

    def __post_init__(self):
        if math.isnan(self.scale):
            # The softmax temperature 1/sqrt(D), held as the float32 value both sides use.
            object.__setattr__(self, "scale", float(np.float32(1.0 / math.sqrt(self.D))))

    @property
    def dtype_code(self) -> int:
        return DTYPE_CODES[self.dtype]

    @property
    def flops(self) -> float:
        """4*B*H*Nq*Nk*D, halved for causal masking."""
        f = 4.0 * self.B * self.H * self.Nq * self.Nk * self.D
        return f / 2 if self.causal else f

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("single_head", 1, 1, 128, 128, 64, "f16", False, seed=1),
        Workload("ragged", 2, 4, 1000, 1000, 64, "f16", False, seed=2),
        Workload("causal_prefill", 1, 32, 2048, 2048, 128, "bf16", True, seed=3),
        Workload("rescale_stress", 4, 32, 4096, 4096, 128, "bf16", False, seed=4,
                 sigma_q=3.0, sigma_k=3.0),
        Workload("long_causal", 1, 16, 16384, 16384, 128, "bf16", True, seed=5),
        Workload("headline", 1, 32, 4096, 4096, 128, "bf16", False, seed=6),
        # a 128-token chunk against a 64K-token context: one query block per head, so the keys
        # are split across CTAs (flash-decoding)
        Workload("long_context_chunk", 1, 8, 128, 65536, 128, "bf16", False, seed=7),
        # the headline shape at head dim 64 (the ragged and single-head configs' D)
        Workload("headline_d64", 1, 32, 4096, 4096, 64, "f16", False, seed=8),
    ]
}


def round_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 array -> uint16 bit patterns of the nearest fp16 / bf16 value (ties to even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = x.view(np.uint32).astype(np.uint64)
        u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
        return u.astype(np.uint16)
    raise ValueError(f"unknown dtype {dtype!r}")


def bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """uint16 bit patterns -> exact float64 values."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def draw(w: Workload) -> dict[str, np.ndarray]:
    """Q [B,H,Nq,D], K and V [B,H,Nk,D] as uint16 bit patterns of w.dtype."""
    sq, sk, sv = np.random.SeedSequence(w.seed).spawn(3)
    out = {}
    for name, ss, shape, sigma in (("q", sq, (w.B, w.H, w.Nq, w.D), w.sigma_q),
                                   ("k", sk, (w.B, w.H, w.Nk, w.D), w.sigma_k),
                                   ("v", sv, (w.B, w.H, w.Nk, w.D), w.sigma_v)):
        x = np.random.default_rng(ss).standard_normal(shape, dtype=np.float32)
        if sigma != 1.0:
            x *= np.float32(sigma)
        out[name] = round_to_bits(x, w.dtype)
    return out


def to_torch(bits: np.ndarray, dtype: str):
    """uint16 bit patterns -> a CPU torch tensor of the matching 16-bit dtype (no copy)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16)


def from_torch(t) -> np.ndarray:
    """A 16-bit torch tensor (any device) -> uint16 bit patterns on the host."""
    import torch

    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
