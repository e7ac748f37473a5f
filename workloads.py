"""Seeded synthetic inputs for FP32 SGEMM, shared by the CUDA path's tests and bench and
by the CPU oracle's tests.

This module holds no GEMM arithmetic. It only draws the operands A (M x K), B (K x N) and
C (M x N) as row-major float32 CPU tensors, in a fixed order from one seeded generator, so
that both sides of every parity check see the same bytes.

Recipe (the generator is not named by any of the pages, so this one is fixed here):
  g = torch.Generator("cpu").manual_seed(seed); draw A, then B, then C, each as float32:
  uniform[-1, 1) is torch.rand(..., generator=g) * 2 - 1, N(0, 1) is torch.randn(...,
  generator=g); "zero" C is torch.zeros and draws nothing. Operands are packed (ld equals
  the number of columns) unless a padded leading dimension is requested, in which case the
  matrix lives in the left columns of a wider buffer and the padding holds a fixed canary.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

CANARY = float("nan")  # value stored in ld padding; any read of it poisons the result


@dataclass(frozen=True)
class Workload:
    """One SGEMM problem: shape, scalars and how its operands are drawn."""

    name: str
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    seed: int
    ab_dist: str  # "uniform" or "normal"
    c_dist: str  # "uniform", "normal" or "zero"
    tags: tuple = field(default_factory=tuple)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


def _draw(shape, dist: str, g: torch.Generator) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float32)
    if dist == "zero":
        return torch.zeros(shape, dtype=torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def _embed(x: torch.Tensor, ld: int) -> torch.Tensor:
    """Place x (rows x cols) in the left columns of a rows x ld buffer filled with CANARY and
    return the strided view (x.stride(0) == ld)."""
    rows, cols = x.shape
    if ld == cols:
        return x.contiguous()
    if ld < cols:
        raise ValueError("leading dimension smaller than the column count")
    buf = torch.full((max(rows, 1), ld), CANARY, dtype=torch.float32)
    buf[:rows, :cols] = x
    return buf[:rows, :cols]


def make_inputs(M: int, N: int, K: int, seed: int, ab_dist: str = "normal",
                c_dist: str = "normal", lda: int | None = None, ldb: int | None = None,
                ldc: int | None = None):
    """Draw (A, B, C) for an M x N x K problem following the module recipe.

    Returns CPU float32 tensors; with a padded ld the tensor is a strided view whose
    stride(0) is that ld."""
    g = torch.Generator("cpu").manual_seed(seed)
    A = _draw((M, K), ab_dist, g)
    B = _draw((K, N), ab_dist, g)
    C = _draw((M, N), c_dist, g)
    return (_embed(A, lda or max(K, 1)), _embed(B, ldb or max(N, 1)),
            _embed(C, ldc or max(N, 1)))


def workload_inputs(w: Workload):
    return make_inputs(w.M, w.N, w.K, w.seed, w.ab_dist, w.c_dist)


# The five benchmark configurations of the FP32 SGEMM study (square, power-of-two versus
# unaligned, headline 8192 cube, and rectangular / ragged / thin shapes). Configuration 5
# re-seeds with 4 for each of its shapes.
CONFIGS = [
    Workload("sgemm_256cube", 256, 256, 256, 1.0, 0.0, 0, "uniform", "uniform", ("small",)),
    Workload("sgemm_1024cube", 1024, 1024, 1024, 1.0, 0.5, 1, "uniform", "uniform"),
    Workload("sgemm_4096cube", 4096, 4096, 4096, 1.0, 0.0, 2, "normal", "zero"),
    Workload("sgemm_4097cube_unaligned", 4097, 4097, 4097, 1.0, 0.0, 2, "normal", "zero"),
    Workload("sgemm_8192cube", 8192, 8192, 8192, 0.5, 2.0, 3, "uniform", "normal",
             ("headline",)),
    Workload("sgemm_8192x14336x4096", 8192, 14336, 4096, 1.0, 1.0, 4, "normal", "normal"),
    Workload("sgemm_4099x3001x777_ragged", 4099, 3001, 777, 1.0, 1.0, 4, "normal", "normal"),
    Workload("sgemm_16x4096x4096_thin_m", 16, 4096, 4096, 1.0, 1.0, 4, "normal", "normal"),
    Workload("sgemm_4096x16x8192_thin_n", 4096, 16, 8192, 1.0, 1.0, 4, "normal", "normal"),
]

BY_NAME = {w.name: w for w in CONFIGS}
HEADLINE = BY_NAME["sgemm_8192cube"]
