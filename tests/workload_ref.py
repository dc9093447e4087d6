"""FP64 oracle results for the full-size workloads, computed once per test process
and shared by the CUDA-core and tensor-core parity checks.

Coverage (the rows of C compared element by element, every column of each row):
  * square256, square1024, square4096: every row, i.e. the whole output;
  * fc8192x4096x11008: 4096 of the 8192 rows -- both sides of every 128-row tile
    boundary, the first and last rows, and a seeded draw for the rest;
  * the batched QK^T and Score x V workloads: the whole first and last problems
    (2 x 2048 rows) and a seeded draw of rows from a few problems in between.
"""

from __future__ import annotations

import functools

import numpy as np

import oracle
from dense_fp32_gemm_sm_gb300 import workloads

FC_ROWS = 4096
BATCH_WHOLE = (0, 127)
BATCH_SAMPLED = {1: 24, 63: 24, 64: 24, 100: 24}


def _fc_rows(M: int, n: int, seed: int) -> np.ndarray:
    edges = {0, 1, M - 2, M - 1}
    for t in range(128, M, 128):
        edges.update((t - 1, t))
    rest = np.setdiff1d(np.arange(M), np.fromiter(edges, np.int64))
    rng = np.random.default_rng(seed)
    extra = rng.choice(rest, size=n - len(edges), replace=False)
    return np.sort(np.concatenate([np.fromiter(edges, np.int64), extra])).astype(np.int64)


def _sampled_rows(M: int, n: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    edges = [0, 1, 127, 128, 255, 256, M // 2, M - 129, M - 128, M - 1]
    extra = rng.choice(M, size=n, replace=False)
    return np.unique(np.concatenate([edges, extra])).astype(np.int64)


@functools.lru_cache(maxsize=None)
def workload(name: str) -> workloads.Workload:
    return workloads.make(name)


@functools.lru_cache(maxsize=None)
def reference(name: str):
    """[(problem index or None, rows, want, mag)] for the workload's checked rows."""
    w = workload(name)
    if w.batch:
        A, B = w.A.numpy(), w.B.numpy()
        parts = []
        plan = [(b, None) for b in BATCH_WHOLE] + [(b, n) for b, n in BATCH_SAMPLED.items()]
        for b, n in plan:
            rows = np.arange(w.M, dtype=np.int64) if n is None else _sampled_rows(w.M, n, b)
            want, mag = oracle.gemm(w.ta, w.tb, w.M, w.N, w.K, w.alpha, A[b].reshape(-1), w.lda,
                                    B[b].reshape(-1), w.ldb, rows=rows)
            parts.append((b, rows, want, mag))
        return parts
    rows = (_fc_rows(w.M, FC_ROWS, seed=3) if w.M > FC_ROWS
            else np.arange(w.M, dtype=np.int64))
    C0 = w.C0.numpy().reshape(-1) if w.C0 is not None else None
    want, mag = oracle.gemm(w.ta, w.tb, w.M, w.N, w.K, w.alpha, w.A.numpy().reshape(-1), w.lda,
                            w.B.numpy().reshape(-1), w.ldb, w.beta, C0, w.ldc, bias=w.bias,
                            relu=w.relu, rows=None if w.M <= FC_ROWS else rows)
    return [(None, rows, want, mag)]


def checked_rows(name: str) -> int:
    return sum(len(rows) for _, rows, _, _ in reference(name))


def compare(name: str, C: np.ndarray, tol: float):
    """Every checked element of C (the library's output, float32) within tol * mag +
    FLT_MIN of the oracle; returns the worst err / (tol * mag + FLT_MIN)."""
    flt_min = float(np.finfo(np.float32).tiny)
    worst = 0.0
    assert not np.isnan(C).any(), "NaN in the output"
    for b, rows, want, mag in reference(name):
        got = (C[b] if b is not None else C)[rows].astype(np.float64)
        bound = tol * mag + flt_min
        ratio = np.abs(got - want) / bound
        bad = ratio > 1.0
        assert not bad.any(), "%s%s: %d of %d elements outside %g*mag, worst ratio %g at %s" % (
            name, "" if b is None else " problem %d" % b, int(bad.sum()), bad.size, tol,
            float(ratio.max()), np.unravel_index(int(ratio.argmax()), ratio.shape))
        worst = max(worst, float(ratio.max()))
    return worst
