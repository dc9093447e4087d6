"""Seeded synthetic inputs for the FP32 GEMM workloads.

This module only draws random numbers; it holds none of the GEMM arithmetic.
Both sides of every parity check (the CUDA library and the CPU oracle) and the
benchmark take their inputs from here, so they see the same bits.

Recipe (the pages give none): a ``torch.Generator('cpu')`` seeded with the
workload's seed draws the tensors in the order the workload lists them, as
float32 and row-major.  ``uniform[lo, hi)`` is ``lo + (hi - lo) * rand`` and
``N(0, s^2)`` is ``s * randn``.  Small-integer inputs (for bit-exact checks)
are ``randint(lo, hi + 1)`` converted to float32.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def uniform(g: torch.Generator, shape, lo: float = -1.0, hi: float = 1.0) -> torch.Tensor:
    return lo + (hi - lo) * torch.rand(*shape, generator=g, dtype=torch.float32)


def normal(g: torch.Generator, shape, std: float = 1.0) -> torch.Tensor:
    return std * torch.randn(*shape, generator=g, dtype=torch.float32)


def small_ints(g: torch.Generator, shape, lo: int = -4, hi: int = 4) -> torch.Tensor:
    return torch.randint(lo, hi + 1, tuple(shape), generator=g).to(torch.float32)


def pooled_ints(g: torch.Generator, count: int, pool: int, width: int, lo: int = -4,
                hi: int = 4):
    """Small-integer rows for a matrix too large to draw element by element: a seeded
    ``pool x width`` block of small integers, then for each of ``count`` rows the index of
    the pool row it repeats.  Returns ``(rows, index)``: row r of the matrix is
    ``rows[index[r]]`` (``index`` is int64)."""
    rows = small_ints(g, (pool, width), lo, hi)
    index = torch.randint(0, pool, (count,), generator=g)
    return rows, index


@dataclass
class Workload:
    """One GEMM problem in the library's argument convention.

    ``A``/``B``/``C0``/``bias`` are CPU float32 tensors holding the operands as
    stored (``A`` is K x M when ``ta`` is 1, ``B`` is N x K when ``tb`` is 1;
    batched operands carry a leading batch dimension).
    """

    name: str
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    ta: int = 0
    tb: int = 0
    batch: int = 0  # 0: a single GEMM; >= 1: strided batch of that many
    relu: bool = False
    seed: int = 0
    A: torch.Tensor | None = field(default=None, repr=False)
    B: torch.Tensor | None = field(default=None, repr=False)
    C0: torch.Tensor | None = field(default=None, repr=False)
    bias: torch.Tensor | None = field(default=None, repr=False)

    @property
    def lda(self) -> int:
        return self.M if self.ta else self.K

    @property
    def ldb(self) -> int:
        return self.K if self.tb else self.N

    @property
    def ldc(self) -> int:
        return self.N

    @property
    def flops(self) -> float:
        """2*M*N*K per problem (GEMM 优化详解, 计算复杂度分析), times the batch."""
        return 2.0 * self.M * self.N * self.K * max(1, self.batch)


# The workloads, smallest first.  Sizes and value distributions follow the pages'
# shapes: square 256/1024/4096 problems, a fully-connected layer Y = ReLU(X W + b),
# batched attention scores S = Q K^T, and the second attention GEMM O = P V.
WORKLOADS = ("square256", "square1024", "square4096", "fc8192x4096x11008", "qkt128x2048x128",
             "pv128x2048x2048x128")


def make(name: str) -> Workload:
    if name == "square256":
        g = generator(0)
        n = 256
        return Workload(name, n, n, n, 1.0, 0.0, seed=0,
                        A=uniform(g, (n, n)), B=uniform(g, (n, n)))
    if name == "square1024":
        g = generator(1)
        n = 1024
        A, B = uniform(g, (n, n)), uniform(g, (n, n))
        return Workload(name, n, n, n, 1.5, 0.5, seed=1, A=A, B=B, C0=uniform(g, (n, n)))
    if name == "square4096":
        g = generator(2)
        n = 4096
        return Workload(name, n, n, n, 1.0, 0.0, seed=2,
                        A=uniform(g, (n, n)), B=uniform(g, (n, n)))
    if name == "fc8192x4096x11008":
        g = generator(3)
        M, K, N = 8192, 4096, 11008
        X = normal(g, (M, K))
        W = normal(g, (K, N), std=1.0 / 64.0)  # variance 1/4096
        b = uniform(g, (N,), -0.1, 0.1)
        return Workload(name, M, N, K, 1.0, 0.0, relu=True, seed=3, A=X, B=W, bias=b)
    if name == "qkt128x2048x128":
        g = generator(4)
        batch, S, D = 128, 2048, 128
        Q = normal(g, (batch, S, D))
        Kt = normal(g, (batch, S, D))
        # alpha = 1/sqrt(128), computed in double and rounded once to float32.
        alpha = float(torch.tensor(1.0 / math.sqrt(D), dtype=torch.float32))
        return Workload(name, S, S, D, alpha, 0.0, ta=0, tb=1, batch=batch, seed=4, A=Q, B=Kt)
    if name == "pv128x2048x2048x128":
        # O = P V per (sequence, head): P 2048 x 2048 attention weights, uniform[0, 1) /
        # 2048 (rows of nonnegative weights summing to about 1/2), V 2048 x 128 ~ N(0, 1).
        g = generator(5)
        batch, S, D = 128, 2048, 128
        P = uniform(g, (batch, S, S), 0.0, 1.0 / S)
        V = normal(g, (batch, S, D))
        return Workload(name, S, D, S, 1.0, 0.0, ta=0, tb=0, batch=batch, seed=5, A=P, B=V)
    raise KeyError("unknown workload %r (known: %s)" % (name, ", ".join(WORKLOADS)))
