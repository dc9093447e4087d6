"""Run one problem through the CUDA library and the FP64 oracle on the same inputs.

Inputs are drawn on the CPU (seeded), stored with padded leading dimensions
(padding holds NaN so any read of it poisons the result) and optionally shifted
by a few elements so pointers are not 16-byte aligned.  The library is called
through its C ABI on device copies; the oracle sees the identical float32 bits.

Acceptance, per output element (fixed by the FP32 accuracy requirement of the
method; the K in "1e-5 * K * sum|A||B| / K" cancels):
    integer-valued inputs:  bit-exact (every partial sum is an integer < 2^24)
    otherwise:              |C - C_ref| <= 1e-5 * mag + FLT_MIN
with mag = |alpha| sum_k |a_ik||b_kj| + |beta||c_ij| + |bias_j| + |row_bias_i| from the
oracle.
Elements of C outside the M x N region must come back unchanged.
"""

from dataclasses import dataclass

import numpy as np
import torch

import dense_fp32_gemm_sm_gb300 as fg
import oracle
from dense_fp32_gemm_sm_gb300 import workloads

REL_TOL = 1e-5
FLT_MIN = float(np.finfo(np.float32).tiny)
SENTINEL = -12345.0


@dataclass
class Case:
    ta: int = 0
    tb: int = 0
    M: int = 64
    N: int = 64
    K: int = 64
    alpha: float = 1.0
    beta: float = 0.0
    batch: int = 0  # 0: single GEMM through gemm_explicit with batch=1
    bias: bool = False
    relu: bool = False
    ints: bool = True
    pad: tuple = (0, 0, 0)  # extra leading-dimension elements for A, B, C
    offset: tuple = (0, 0, 0)  # element offset of A, B, C from a 16-byte boundary
    config: int = -1
    seed: int = 0
    align_ld: bool = True  # round leading dimensions and batch strides up to 16 bytes
    math: int = -1  # >= 0: call fgemm_gemm_math with this arithmetic instead of gemm_explicit
    c_nan: bool = False  # fill the initial C with NaN (only meaningful for beta == 0)
    a_nan: bool = False  # fill A with NaN (only meaningful for alpha == 0)
    row_bias: bool = False  # call fgemm_sgemm_row_bias_relu with a per-row bias (single GEMM)
    # With a tensor-core math: whether the call must run on the tensor cores (True) or
    # fall back to the CUDA-core kernel (False), as fgemm_math_supported reports; None
    # leaves it open (random cases whose alignment may go either way).
    expect_tc: object = True
    # Not None: call fgemm_sgemm_staged with this stage argument (-1: the model's choice,
    # 0..3: the operands to copy k-major) and a NaN-filled workspace of the size
    # fgemm_staged_workspace_size gives; with math >= 0, fgemm_gemm_math_staged and a
    # workspace of fgemm_math_staged_workspace_size.
    stage: object = None
    share_a: bool = False  # batch stride 0 for A (every problem reads the same A)
    share_b: bool = False
    # (operand "A" or "B", stored row, stored column, value): entries set in every problem
    # after the draw -- IEEE special values (NaN, +-Inf) among the small integers.
    specials: tuple = ()


def _draw(g, shape, ints):
    if ints:
        return workloads.small_ints(g, shape).numpy()
    return workloads.uniform(g, shape).numpy()


def _device(flat, offset):
    """Copy a flat float32 array to the GPU at `offset` elements past a 256-byte boundary."""
    buf = torch.empty(flat.size + offset + 4, dtype=torch.float32, device="cuda")
    buf[offset:offset + flat.size].copy_(torch.from_numpy(flat))
    return buf, buf.data_ptr() + 4 * offset


def run(case: Case):
    """Returns (got, want, mag, untouched_ok) with got/want of shape (batch or 1, M, N)."""
    g = workloads.generator(case.seed)
    nb = max(case.batch, 1)
    M, N, K = case.M, case.N, case.K
    up = (lambda x: (x + 3) // 4 * 4) if case.align_ld else (lambda x: x)
    lda = up(max(1, (M if case.ta else K) + case.pad[0]))
    ldb = up(max(1, (K if case.tb else N) + case.pad[1]))
    ldc = up(max(1, N + case.pad[2]))
    a_rows, b_rows = (K if case.ta else M), (N if case.tb else K)
    sA, sB, sC = up(a_rows * lda + 3), up(b_rows * ldb + 5), up(M * ldc + 7)
    if case.batch == 0:
        sA = sB = sC = 0
    if case.share_a:
        sA = 0
    if case.share_b:
        sB = 0

    def stored(rows, ld, cols, stride, ints):
        flat = np.full(max(stride * (nb - 1) + rows * ld, 1), np.nan, np.float32)
        for b in range(nb):
            blk = _draw(g, (rows, cols), ints)
            for r in range(rows):
                flat[b * stride + r * ld: b * stride + r * ld + cols] = blk[r]
        return flat

    A = stored(a_rows, lda, M if case.ta else K, sA, case.ints)
    B = stored(b_rows, ldb, K if case.tb else N, sB, case.ints)
    C0 = stored(M, ldc, N, sC, True)
    # padding of C holds a sentinel that must survive the call
    C0[np.isnan(C0)] = SENTINEL
    if case.c_nan:
        for b in range(nb):
            for r in range(M):
                C0[b * sC + r * ldc: b * sC + r * ldc + N] = np.nan
    for which, r, c, v in case.specials:
        flat, ld, stride = (A, lda, sA) if which == "A" else (B, ldb, sB)
        for b in range(nb):
            flat[b * stride + r * ld + c] = v
    if case.a_nan:
        A[:] = np.nan
    bias = _draw(g, (N,), True).astype(np.float32) if case.bias else None
    row_bias = _draw(g, (M,), True).astype(np.float32) if case.row_bias else None
    if row_bias is not None:
        assert case.batch == 0 and case.math < 0 and case.config < 0 and bias is None

    dA, pA = _device(A, case.offset[0])
    dB, pB = _device(B, case.offset[1])
    dC, pC = _device(C0, case.offset[2])
    dbias, pbias = _device(bias, 0) if bias is not None else (None, None)
    drow, prow = _device(row_bias, 0) if row_bias is not None else (None, None)
    stream = torch.cuda.current_stream().cuda_stream
    if row_bias is not None:
        fg.sgemm_row_bias_relu(case.ta, case.tb, M, N, K, case.alpha, pA, lda, pB, ldb, case.beta,
                               pC, ldc, prow, case.relu, stream=stream)
    elif case.math >= 0 and case.stage is not None:
        ws_bytes = fg.math_staged_workspace_size(case.math, case.ta, case.tb, M, N, K, nb)
        ws = torch.full((ws_bytes // 4 + 1,), float("nan"), device="cuda")
        fg.gemm_math_staged(case.math, case.ta, case.tb, M, N, K, case.alpha, pA, lda, sA, pB,
                            ldb, sB, case.beta, pC, ldc, sC, nb, pbias, case.relu, case.stage, ws,
                            ws_bytes, stream=stream)
    elif case.math >= 0:
        if case.math != fg.MATH_FP32 and case.expect_tc is not None:
            path = fg.math_supported(case.math, case.ta, case.tb, M, N, K, case.alpha, pA, lda, sA,
                                     pB, ldb, sB, nb)
            assert path == (1 if case.expect_tc else 0), (
                "fgemm_math_supported says %d, the case expects %s" % (
                    path, "the tensor cores" if case.expect_tc else "the CUDA-core fallback"))
        fg.gemm_math(case.math, case.ta, case.tb, M, N, K, case.alpha, pA, lda, sA, pB, ldb, sB,
                     case.beta, pC, ldc, sC, nb, pbias, case.relu, stream=stream)
    elif case.stage is not None:
        assert case.config < 0
        ws_bytes = fg.staged_workspace_size(case.ta, case.tb, M, N, K, nb)
        ws = torch.full((ws_bytes // 4 + 1,), float("nan"), device="cuda")
        fg.sgemm_staged(case.ta, case.tb, M, N, K, case.alpha, pA, lda, sA, pB, ldb, sB,
                        case.beta, pC, ldc, sC, nb, pbias, case.relu, case.stage, ws, ws_bytes,
                        stream=stream)
    else:
        fg.gemm_explicit(case.config, case.ta, case.tb, M, N, K, case.alpha, pA, lda, sA, pB, ldb,
                         sB, case.beta, pC, ldc, sC, nb, pbias, case.relu, stream=stream)
    torch.cuda.synchronize()
    assert fg.device_status() == fg.OK, "a tensor-core wait ran out"
    Cout = dC[case.offset[2]:case.offset[2] + C0.size].cpu().numpy()

    got = np.zeros((nb, M, N), np.float32)
    want = np.zeros((nb, M, N), np.float64)
    mag = np.zeros((nb, M, N), np.float64)
    untouched = np.ones(C0.size, bool)
    for b in range(nb):
        o, m = oracle.gemm(case.ta, case.tb, M, N, K, case.alpha, A[b * sA:], lda, B[b * sB:],
                           ldb, case.beta, C0[b * sC:] if case.beta != 0 else None, ldc,
                           bias=bias, relu=case.relu, row_bias=row_bias)
        want[b], mag[b] = o, m
        for r in range(M):
            got[b, r] = Cout[b * sC + r * ldc: b * sC + r * ldc + N]
            untouched[b * sC + r * ldc: b * sC + r * ldc + N] = False
    same = (Cout == C0) | (np.isnan(Cout) & np.isnan(C0))
    return got, want, mag, bool(same[untouched].all())


def check(case: Case, rel_tol=REL_TOL):
    got, want, mag, untouched_ok = run(case)
    assert untouched_ok, "the call wrote outside the M x N region of C"
    assert not np.isnan(got).any(), "NaN in the result"
    if case.ints:
        bad = got.astype(np.float64) != want
        assert not bad.any(), "not bit-exact: %d of %d differ, first at %s: %r vs %r" % (
            bad.sum(), bad.size, np.argwhere(bad)[0], got[bad][0], want[bad][0])
    else:
        err = np.abs(got.astype(np.float64) - want)
        bound = rel_tol * mag + FLT_MIN
        bad = err > bound
        assert not bad.any(), "outside %g*mag: %d of %d, worst ratio %g" % (
            rel_tol, bad.sum(), bad.size, (err / bound).max())
    return float((np.abs(got.astype(np.float64) - want) / (mag + FLT_MIN)).max())
