"""Seeded synthetic GEMM inputs.

This module only draws random operands; it holds none of the GEMM
arithmetic, and both the CPU oracle's tests and the CUDA path's tests and
benchmark take their inputs from it.

Recipe (the pages use no public dataset; every input is synthetic):
  * one ``torch.Generator('cpu')`` per workload, seeded with the workload's
    seed; A (M x K) is drawn first, then B (K x N), both as float32;
  * "uniform":  ``rand * 2 - 1``           (i.i.d. uniform on [-1, 1));
  * "normal":   ``randn / sqrt(K)``        (i.i.d. normal(0, 1) / sqrt(K));
  * "int":      ``randint(lo, hi + 1)``    (integer values, exact in every type);
  * the float32 draw is then cast to the workload's type with torch's
    round-to-nearest-even cast (FP16 / BF16); the oracle sees the cast values.
Operands are row-major with lda = K, ldb = N, ldc = N unless a test builds a
strided view on purpose.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str          # "f32" | "f16" | "bf16"
    M: int
    N: int
    K: int
    dist: str           # "uniform" | "normal" | "int"
    seed: int
    lo: int = -2        # integer range for dist == "int"
    hi: int = 2

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def with_shape(self, M: int, N: int, K: int, name: str | None = None) -> "Workload":
        return replace(self, M=M, N=N, K=K, name=name or f"{self.name}_{M}x{N}x{K}")


# The seeded workloads of the GEMM benchmark suite.
WORKLOADS = {
    w.name: w for w in [
        Workload("f32_256", "f32", 256, 256, 256, "uniform", 0),
        # integer-valued copy of the 256^3 case: |partial sums| <= 4*256 < 2^24
        Workload("f32_256_int", "f32", 256, 256, 256, "int", 100, -2, 2),
        Workload("f32_2048", "f32", 2048, 2048, 2048, "uniform", 1),
        Workload("f32_4096", "f32", 4096, 4096, 4096, "uniform", 2),
        Workload("f16_4096", "f16", 4096, 4096, 4096, "normal", 3),
        Workload("bf16_8192", "bf16", 8192, 8192, 8192, "normal", 3),
        Workload("f32_edge", "f32", 1000, 1030, 777, "uniform", 4),
        Workload("bf16_edge", "bf16", 4097, 3000, 1536, "uniform", 4),
        # a skinny product (two output tiles, long K): single CTAs, split-K
        Workload("f16_skinny", "f16", 256, 256, 65536, "normal", 5),
    ]
}


def _draw(shape, w: Workload, g: torch.Generator) -> torch.Tensor:
    if w.dist == "uniform":
        x = torch.rand(shape, generator=g, dtype=torch.float32) * 2 - 1
    elif w.dist == "normal":
        x = torch.randn(shape, generator=g, dtype=torch.float32) / math.sqrt(max(w.K, 1))
    elif w.dist == "int":
        x = torch.randint(w.lo, w.hi + 1, shape, generator=g).to(torch.float32)
    else:
        raise ValueError(f"unknown distribution {w.dist!r}")
    return x.to(TORCH_DTYPES[w.dtype])


def make(w: Workload | str):
    """Return (A, B) as contiguous CPU tensors of the workload's dtype."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    g = torch.Generator("cpu")
    g.manual_seed(w.seed)
    A = _draw((w.M, w.K), w, g)
    B = _draw((w.K, w.N), w, g)
    return A, B


def to_numpy_bits(t: torch.Tensor) -> np.ndarray:
    """CPU tensor -> numpy array the oracle takes: float32 as is, FP16/BF16 as
    uint16 bit patterns (same memory layout, strides preserved)."""
    t = t.detach().cpu()
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16)
    raise TypeError(f"unsupported dtype {t.dtype}")


def sample_rows(M: int, count: int, seed: int, tile: int = 128) -> np.ndarray:
    """Deterministic sample of output rows: the first and last row, the rows
    on both sides of every few tile boundaries, and random rows."""
    rng = np.random.default_rng(seed)
    fixed = {0, M - 1}
    for b in range(tile, M, tile * max(1, (M // tile) // 4 or 1)):
        fixed.update({b - 1, b})
    fixed.update(int(r) for r in rng.integers(0, M, size=max(0, count - len(fixed))))
    return np.array(sorted(r for r in fixed if 0 <= r < M), dtype=np.int64)
