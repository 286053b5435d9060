"""Seeded synthetic inputs for the mixed-precision GEMM, shared by the oracle
side and the CUDA side.

This module only draws numbers and lays them out in memory; it holds none of
the GEMM's arithmetic. The five named workloads and their value
distributions follow the benchmark shapes of the project; the pages' own
harness conventions they rely on are:

* "Day 80, Capstone 4: a tensor-core GEMM", "Independent gate": symmetric
  uniform, normal and exact small-integer inputs, ragged sizes such as
  611 x 613 x 617 and K = 617 ("Faded practice", practice 3).
* "Day 72: Tensor cores with WMMA", "Why this program calls cuBLAS twice":
  small integers in [-3, 3] (A) and [-2, 2] (B), exact in FP16.
* "GEMM kernels 1-7 + Tensor Cores", side-by-side table: the M = 1000,
  K = 1200, N = 800 shape.

Every value is drawn in float32 from a CPU ``torch.Generator`` and rounded to
FP16 with ``.half()`` (round to nearest even); only the resulting FP16 bits
matter, and both sides read the same bits. Padding columns beyond K (A) or
N (B) when the leading dimension is larger are filled with FP16 NaN, and the
padding of C beyond N with float32 NaN, so a kernel that reads or writes past
the logical extent is caught.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

FP16_NAN_BITS = 0x7E00


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    lda: int
    ldb: int
    ldc: int
    alpha: float
    beta: float
    dist: str          # distribution of A and B
    c_dist: str        # distribution of the incoming C ("zeros" when beta == 0)
    seed_base: int
    full_check: bool   # every element checked, else a seeded sample plus edges

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


WORKLOADS = {
    0: Workload("ragged_tiny_200x136x617", 200, 136, 617, 617, 136, 136, 1.0, 0.0,
                "uniform", "zeros", 1000, True),
    1: Workload("square_2048", 2048, 2048, 2048, 2048, 2048, 2048, 1.0, 0.0,
                "uniform", "zeros", 1010, True),
    2: Workload("ragged_1000x800x1200", 1000, 800, 1200, 1200, 800, 800, 1.5, 1.0,
                "normal_clip4", "normal", 1020, True),
    3: Workload("square_8192", 8192, 8192, 8192, 8192, 8192, 8192, 1.0, 0.0,
                "normal_0.5", "zeros", 1030, False),
    4: Workload("tall_skinny_65536x257x4093", 65536, 257, 4093, 4093, 257, 257, 1.0, 0.5,
                "uniform", "uniform", 1040, False),
}


def _draw(gen: torch.Generator, shape, dist: str) -> torch.Tensor:
    if dist == "uniform":            # uniform[-1, 1)
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal":             # N(0, 1)
        return torch.randn(shape, generator=gen, dtype=torch.float32)
    if dist == "normal_clip4":       # N(0, 1) clipped to [-4, 4]
        return torch.randn(shape, generator=gen, dtype=torch.float32).clamp_(-4.0, 4.0)
    if dist == "normal_0.5":         # N(0, 0.5^2)
        return torch.randn(shape, generator=gen, dtype=torch.float32) * 0.5
    if dist == "int3":               # integers in [-3, 3]
        return torch.randint(-3, 4, shape, generator=gen).to(torch.float32)
    if dist == "int2":               # integers in [-2, 2]
        return torch.randint(-2, 3, shape, generator=gen).to(torch.float32)
    if dist == "ones":
        return torch.ones(shape, dtype=torch.float32)
    if dist == "zeros":
        return torch.zeros(shape, dtype=torch.float32)
    if dist == "subnormal":          # integers in [-1023, 1023] times 2^-24: FP16 subnormals (or 0)
        return torch.randint(-1023, 1024, shape, generator=gen).to(torch.float32) * 2.0 ** -24
    if dist == "int3_x8192":         # integers in [-3, 3] times 2^13
        return torch.randint(-3, 4, shape, generator=gen).to(torch.float32) * 8192.0
    if dist == "edge":               # magnitudes near the top of the FP16 range
        mag = 32768.0 + torch.rand(shape, generator=gen, dtype=torch.float32) * 32736.0
        sign = torch.randint(0, 2, shape, generator=gen).to(torch.float32) * 2.0 - 1.0
        return mag * sign
    raise ValueError(f"unknown distribution {dist!r}")


def _padded(values: torch.Tensor, rows: int, cols: int, ld: int, fill) -> torch.Tensor:
    if ld == cols:
        return values.contiguous()
    out = torch.full((rows, ld), fill, dtype=values.dtype)
    out[:, :cols] = values
    return out


@dataclasses.dataclass
class Operands:
    """Host operands: A [M, lda] fp16, B [K, ldb] fp16 (or [N, ldb] when
    b_col_major: row j holds column j of B), C [M, ldc] fp32."""
    M: int
    N: int
    K: int
    lda: int
    ldb: int
    ldc: int
    alpha: float
    beta: float
    A: torch.Tensor
    B: torch.Tensor
    C: torch.Tensor
    b_col_major: bool = False

    def bits(self, name: str) -> np.ndarray:
        """Flat numpy view of an operand (uint16 bit patterns for A and B)."""
        t = getattr(self, name)
        if t.dtype == torch.float16:
            return t.reshape(-1).view(torch.int16).numpy().view(np.uint16)
        return t.reshape(-1).numpy()


def make_operands(M: int, N: int, K: int, *, lda: Optional[int] = None, ldb: Optional[int] = None,
                  ldc: Optional[int] = None, alpha: float = 1.0, beta: float = 0.0,
                  dist: str = "uniform", dist_b: Optional[str] = None, c_dist: str = "zeros",
                  seed: int = 0, b_col_major: bool = False) -> Operands:
    """Seeded operands; A uses ``seed``, B ``seed + 1``, C ``seed + 2``. With
    ``b_col_major`` the same values of B are stored column by column."""
    lda = max(K, 1) if lda is None else lda
    ldb = max(K if b_col_major else N, 1) if ldb is None else ldb
    ldc = max(N, 1) if ldc is None else ldc
    ga = torch.Generator().manual_seed(seed)
    gb = torch.Generator().manual_seed(seed + 1)
    gc = torch.Generator().manual_seed(seed + 2)
    a = _draw(ga, (M, K), dist).half()
    b = _draw(gb, (K, N), dist_b or dist).half()
    c = _draw(gc, (M, N), c_dist)
    nan16 = torch.tensor([FP16_NAN_BITS], dtype=torch.int16).view(torch.float16).item()
    A = _padded(a, M, K, lda, nan16)
    B = _padded(b.t().contiguous(), N, K, ldb, nan16) if b_col_major else _padded(b, K, N, ldb, nan16)
    C = _padded(c, M, N, ldc, float("nan"))
    return Operands(M, N, K, lda, ldb, ldc, alpha, beta, A, B, C, b_col_major)


def workload_operands(index: int) -> Operands:
    w = WORKLOADS[index]
    return make_operands(w.M, w.N, w.K, lda=w.lda, ldb=w.ldb, ldc=w.ldc, alpha=w.alpha,
                         beta=w.beta, dist=w.dist, c_dist=w.c_dist, seed=w.seed_base)


def sample_indices(M: int, N: int, count: int, seed: int, edges: bool = True):
    """``count`` seeded random (i, j) plus, if ``edges``, every element of rows
    0 and M-1 and columns 0 and N-1. Returns two int64 arrays."""
    g = torch.Generator().manual_seed(seed)
    I = torch.randint(0, M, (count,), generator=g, dtype=torch.int64)
    J = torch.randint(0, N, (count,), generator=g, dtype=torch.int64)
    parts_i, parts_j = [I], [J]
    if edges:
        cols = torch.arange(N, dtype=torch.int64)
        rows = torch.arange(M, dtype=torch.int64)
        for r in sorted({0, M - 1}):
            parts_i.append(torch.full((N,), r, dtype=torch.int64)); parts_j.append(cols)
        for c in sorted({0, N - 1}):
            parts_i.append(rows); parts_j.append(torch.full((M,), c, dtype=torch.int64))
    return torch.cat(parts_i).numpy(), torch.cat(parts_j).numpy()


def workload_sample(index: int, count: int = 65536):
    w = WORKLOADS[index]
    return sample_indices(w.M, w.N, count, w.seed_base + 3)
