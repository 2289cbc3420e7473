"""Seeded synthetic inputs shaped like LLM GEMM operands.

Shared by the tests, the benchmark and the oracle's callers. This module holds
no quantisation arithmetic: it only draws FP32 values with torch's CPU generator
and rounds them once to BF16 (nearest-even), so that every consumer reads the
same bits.

Workloads (shapes, distributions and seeds):
  act_small   1024 x 1024, N(0,1), exactly round(0.005 N) distinct positions x 20
  activation  8192 x 4096, Student-t (nu = 3) times a per-column lognormal(0,1) scale
  gradient    4096 x 14336 and 14336 x 4096, N(0, 1e-3^2), round(0.001 N) positions x 100
  sweep       R x 4096 N(0,1), R = 2^8 .. 2^18
  gemm        A, B 8192 x 8192, N(0, 1/8192)
"""
from __future__ import annotations

import math

import torch

SEEDS = {"act_small": 101, "activation": 102, "grad_a": 103, "grad_b": 104,
         "sweep": 105, "gemm_a": 106, "gemm_b": 107}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal_with_outliers(rows: int, cols: int, std: float, frac: float, mult: float,
                         seed: int) -> torch.Tensor:
    """N(0, std^2) with exactly round(frac * rows * cols) distinct positions
    (a seeded random permutation) multiplied by ``mult``; BF16."""
    g = _gen(seed)
    x = torch.randn(rows, cols, generator=g, dtype=torch.float32) * std
    n = rows * cols
    k = int(round(frac * n))
    if k:
        pos = torch.randperm(n, generator=g)[:k]
        x.view(-1)[pos] *= mult
    return x.to(torch.bfloat16)


def student_t_colscaled(rows: int, cols: int, nu: int, seed: int) -> torch.Tensor:
    """Student-t with ``nu`` degrees of freedom drawn as Z / sqrt(V / nu), V a
    sum of ``nu`` squared standard normals, times a per-column exp(N(0,1));
    BF16."""
    g = _gen(seed)
    z = torch.randn(rows, cols, generator=g, dtype=torch.float32)
    v = torch.zeros(rows, cols, dtype=torch.float32)
    for _ in range(nu):
        n = torch.randn(rows, cols, generator=g, dtype=torch.float32)
        v += n * n
    t = z / torch.sqrt(v / nu)
    col = torch.exp(torch.randn(1, cols, generator=g, dtype=torch.float32))
    return (t * col).to(torch.bfloat16)


def normal(rows: int, cols: int, std: float, seed: int) -> torch.Tensor:
    g = _gen(seed)
    return (torch.randn(rows, cols, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


# ---- the named workloads ---------------------------------------------------

def act_small() -> torch.Tensor:
    return normal_with_outliers(1024, 1024, 1.0, 0.005, 20.0, SEEDS["act_small"])


def activation(rows: int = 8192, cols: int = 4096) -> torch.Tensor:
    return student_t_colscaled(rows, cols, 3, SEEDS["activation"])


def gradient(which: str = "a", rows: int | None = None, cols: int | None = None) -> torch.Tensor:
    if which == "a":
        r, c, s = rows or 4096, cols or 14336, SEEDS["grad_a"]
    else:
        r, c, s = rows or 14336, cols or 4096, SEEDS["grad_b"]
    return normal_with_outliers(r, c, 1e-3, 0.001, 100.0, s)


def sweep(rows: int, cols: int = 4096) -> torch.Tensor:
    return normal(rows, cols, 1.0, SEEDS["sweep"])


def sweep_rows() -> list[int]:
    return [2 ** p for p in range(8, 19)]


def gemm_operand(which: str = "a", n: int = 8192, k: int = 8192) -> torch.Tensor:
    seed = SEEDS["gemm_a"] if which == "a" else SEEDS["gemm_b"]
    return normal(n, k, 1.0 / math.sqrt(k), seed)


def bf16_bits(x: torch.Tensor):
    """numpy uint16 view of a BF16 CPU tensor (the oracle's input form)."""
    import numpy as np
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)
