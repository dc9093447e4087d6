"""Pins for the FP64 oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with a hand-worked example, a closed form, an
invariant of the definition, or a library routine on a special case.  They are
plain functions so the same set can be run against deliberately broken copies
of the oracle (tests/test_oracle_mutants.py) to show that a plausible mistake
anywhere in it fails at least one of them.

Definitions pinned (page title, section):
  GEMM 优化详解, "数学定义":            C = alpha*A*B + beta*C
  第5章-基础Kernel, "1.1 什么是矩阵乘法": C[i][j] = sum_{k=0}^{K-1} A[i][k]*B[k][j]
  第5章-基础Kernel, "3.2 分块策略可视化": C00 = A00*B00 + A01*B10 (tile decomposition)
  GEMM 优化详解, "Level 6: Kernel Fusion": relu(acc + bias[col])
"""

import itertools

import numpy as np
import torch

import golden_io
from layout import store

COMBOS = list(itertools.product((0, 1), (0, 1)))


def _run(orc, A_log, B_log, ta, tb, alpha=1.0, beta=0.0, C0=None, bias=None, relu=False,
         pad=(0, 0, 0), fill=np.nan, row_bias=None, **kw):
    """Call the oracle on logical operands stored with transposes and padded ld."""
    M, K = A_log.shape
    N = B_log.shape[1]
    lda = (M if ta else K) + pad[0]
    ldb = (K if tb else N) + pad[1]
    ldc = N + pad[2]
    lda, ldb, ldc = max(lda, 1), max(ldb, 1), max(ldc, 1)
    A = store(A_log, ta, lda, fill) if M * K else None
    B = store(B_log, tb, ldb, fill) if K * N else None
    C0s = store(C0, 0, ldc, fill) if C0 is not None else None
    return orc.gemm(ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C0s, ldc,
                    bias=None if bias is None else np.asarray(bias, np.float32), relu=relu,
                    row_bias=None if row_bias is None else np.asarray(row_bias, np.float32), **kw)


def _exact(got, want, what):
    got, want = np.asarray(got), np.asarray(want)
    assert got.shape == want.shape, "%s: shape %s vs %s" % (what, got.shape, want.shape)
    bad = ~((got == want) | (np.isnan(got) & np.isnan(want)))
    assert not bad.any(), "%s: %d mismatches, first at %s: %r vs %r" % (
        what, bad.sum(), np.argwhere(bad)[0], got[bad][0], want[bad][0])


def pin_golden(orc):
    """Hand-worked 2x2 and 4x4 examples, in every transpose combination, with padded ld."""
    for fname in ("gemm_2x2.txt", "gemm_4x4.txt"):
        for case in golden_io.load(fname):
            for ta, tb in COMBOS:
                for pad in ((0, 0, 0), (3, 1, 2)):
                    out, mag = _run(orc, case["A"], case["B"], ta, tb, case["alpha"], case["beta"],
                                    case.get("C0"), case.get("bias"), case["relu"], pad=pad,
                                    row_bias=case.get("row_bias"))
                    tag = "%s %s ta=%d tb=%d pad=%s" % (fname, case["name"], ta, tb, pad)
                    _exact(out, case["expect"], tag)
                    _exact(mag, case["mag"], tag + " mag")


def pin_ones(orc):
    """ones(M,K) @ ones(K,N) = K everywhere (closed form)."""
    for (M, N, K) in ((3, 5, 7), (8, 1, 33), (1, 1, 1), (5, 6, 1000)):
        for ta, tb in COMBOS:
            out, mag = _run(orc, np.ones((M, K)), np.ones((K, N)), ta, tb, pad=(1, 2, 0))
            _exact(out, np.full((M, N), float(K)), "ones %s" % ((M, N, K, ta, tb),))
            _exact(mag, np.full((M, N), float(K)), "ones mag")


def pin_identity(orc):
    """A @ I = A and I @ B = B exactly (a single nonzero term per sum)."""
    rng = np.random.default_rng(11)
    A = rng.uniform(-1, 1, (7, 5)).astype(np.float32)
    B = rng.uniform(-1, 1, (5, 9)).astype(np.float32)
    for ta, tb in COMBOS:
        out, _ = _run(orc, A, np.eye(5), ta, tb, pad=(2, 1, 3))
        _exact(out, A.astype(np.float64), "A@I ta=%d tb=%d" % (ta, tb))
        out, _ = _run(orc, np.eye(5), B, ta, tb, pad=(0, 2, 1))
        _exact(out, B.astype(np.float64), "I@B ta=%d tb=%d" % (ta, tb))


def pin_index_ramps(orc):
    """Ramps in one index at a time: C[i][j] = K*j, = K*i, = K(K-1)/2 (closed forms)."""
    M, N, K = 6, 7, 9
    cols = np.tile(np.arange(N, dtype=np.float64), (K, 1))  # B[k][j] = j
    rows = np.tile(np.arange(M, dtype=np.float64)[:, None], (1, K))  # A[i][k] = i
    kk_a = np.tile(np.arange(K, dtype=np.float64), (M, 1))  # A[i][k] = k
    kk_b = np.tile(np.arange(K, dtype=np.float64)[:, None], (1, N))  # B[k][j] = k
    for ta, tb in COMBOS:
        out, _ = _run(orc, np.ones((M, K)), cols, ta, tb, pad=(1, 1, 1))
        _exact(out, np.tile(K * np.arange(N, dtype=np.float64), (M, 1)), "K*j")
        out, _ = _run(orc, rows, np.ones((K, N)), ta, tb, pad=(1, 1, 1))
        _exact(out, np.tile(K * np.arange(M, dtype=np.float64)[:, None], (1, N)), "K*i")
        out, _ = _run(orc, kk_a, np.ones((K, N)), ta, tb)
        _exact(out, np.full((M, N), K * (K - 1) / 2.0), "sum k (A)")
        out, _ = _run(orc, np.ones((M, K)), kk_b, ta, tb)
        _exact(out, np.full((M, N), K * (K - 1) / 2.0), "sum k (B)")


def pin_zero_operands(orc):
    """A = 0 gives C = beta*C0 exactly; with bias and ReLU, max(0, beta*C0 + b)."""
    rng = np.random.default_rng(5)
    M, N, K = 5, 6, 4
    C0 = rng.integers(-3, 4, (M, N)).astype(np.float32)
    b = rng.integers(-3, 4, N).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    for ta, tb in COMBOS:
        out, _ = _run(orc, np.zeros((M, K)), B, ta, tb, 1.0, -2.0, C0)
        _exact(out, -2.0 * C0.astype(np.float64), "zero A, beta=-2")
        out, _ = _run(orc, np.zeros((M, K)), B, ta, tb, 1.0, 0.0, None, b, True)
        _exact(out, np.tile(np.maximum(b, 0).astype(np.float64), (M, 1)), "zero A, bias+relu")


def pin_k_zero(orc):
    """K = 0: no products; C = beta*C0 (+ bias, ReLU), and A, B are never read."""
    M, N = 4, 3
    C0 = np.arange(M * N, dtype=np.float32).reshape(M, N) - 5
    b = np.array([1, -20, 3], np.float32)
    out, mag = orc.gemm(0, 0, M, N, 0, 3.0, None, 1, None, N, 0.5, C0.reshape(-1), N)
    _exact(out, 0.5 * C0.astype(np.float64), "K=0")
    _exact(mag, 0.5 * np.abs(C0).astype(np.float64), "K=0 mag")
    out, _ = orc.gemm(1, 1, M, N, 0, 1.0, None, M, None, 1, 1.0, C0.reshape(-1), N,
                      bias=b, relu=True)
    _exact(out, np.maximum(C0 + b, 0).astype(np.float64), "K=0 bias relu")


def pin_unread_operands(orc):
    """beta = 0 never reads C0 (NaN stays out); alpha = 0 never reads A or B."""
    rng = np.random.default_rng(6)
    A = rng.integers(-3, 4, (3, 4)).astype(np.float32)
    B = rng.integers(-3, 4, (4, 5)).astype(np.float32)
    nanC = np.full(15, np.nan, np.float32)
    out, _ = orc.gemm(0, 0, 3, 5, 4, 1.0, A.reshape(-1), 4, B.reshape(-1), 5, 0.0, nanC, 5)
    _exact(out, (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64), "beta=0")
    infA = np.full(12, np.inf, np.float32)
    C0 = np.arange(15, dtype=np.float32)
    out, _ = orc.gemm(0, 0, 3, 5, 4, 0.0, infA, 4, B.reshape(-1), 5, 2.0, C0, 5)
    _exact(out, 2.0 * C0.reshape(3, 5).astype(np.float64), "alpha=0")


def pin_linearity(orc):
    """oracle(alpha, beta) = alpha*oracle(1, 0) + beta*C0 to a few ulp of double."""
    rng = np.random.default_rng(7)
    M, N, K = 9, 11, 37
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    C0 = rng.uniform(-1, 1, (M, N)).astype(np.float32)
    for ta, tb in COMBOS:
        base, mag1 = _run(orc, A, B, ta, tb)
        for alpha, beta in ((1.5, 0.5), (-0.75, 2.0), (3.0, -1.0)):
            out, mag = _run(orc, A, B, ta, tb, alpha, beta, C0, pad=(2, 0, 1))
            want = alpha * base + beta * C0.astype(np.float64)
            assert np.all(np.abs(out - want) <= 8 * np.finfo(np.float64).eps * (mag + 1e-300)), \
                "linearity alpha=%g beta=%g" % (alpha, beta)
            _exact(mag, abs(alpha) * mag1 + abs(beta) * np.abs(C0).astype(np.float64),
                   "linearity mag")


def pin_transpose_identity(orc):
    """(A B)^T = B^T A^T: the transposed call, stored N x M, equals the plain one."""
    rng = np.random.default_rng(8)
    M, N, K = 7, 10, 13
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    out, mag = orc.gemm(0, 0, M, N, K, 1.0, A.reshape(-1), K, B.reshape(-1), N)
    # op(A') = B^T from B's own storage (ta=1), op(B') = A^T from A's storage (tb=1).
    outT, magT = orc.gemm(1, 1, N, M, K, 1.0, B.reshape(-1), N, A.reshape(-1), K)
    _exact(outT, out.T, "(AB)^T = B^T A^T")
    _exact(magT, mag.T, "(AB)^T mag")
    for ta, tb in COMBOS:
        o, _ = _run(orc, B.T, A.T, ta, tb, pad=(1, 2, 3))
        _exact(o, out.T, "B^T A^T ta=%d tb=%d" % (ta, tb))


def pin_block_decomposition(orc):
    """4x4 split into 2x2 tiles: C00 = A00 B00 + A01 B10 (integer data, exact),
    accumulated through beta = 1 and sub-matrix views with leading dimension 4."""
    rng = np.random.default_rng(9)
    A = rng.integers(-4, 5, (4, 4)).astype(np.float32)
    B = rng.integers(-4, 5, (4, 4)).astype(np.float32)
    full, _ = orc.gemm(0, 0, 4, 4, 4, 1.0, A.reshape(-1), 4, B.reshape(-1), 4)
    Af, Bf = A.reshape(-1), B.reshape(-1)
    for bi in (0, 1):
        for bj in (0, 1):
            acc = np.zeros(2 * 4, np.float32)  # a 2x2 tile with ldc 4
            for bk in (0, 1):
                a_view = Af[(2 * bi) * 4 + 2 * bk:]
                b_view = Bf[(2 * bk) * 4 + 2 * bj:]
                part, _ = orc.gemm(0, 0, 2, 2, 2, 1.0, a_view, 4, b_view, 4, 1.0, acc, 4)
                acc[0:2] = part[0]
                acc[4:6] = part[1]
            tile = np.array([acc[0:2], acc[4:6]], np.float64)
            _exact(tile, full[2 * bi:2 * bi + 2, 2 * bj:2 * bj + 2], "C%d%d tiles" % (bi, bj))


def pin_integer_exact(orc):
    """Small-integer data: the result is an exact integer, equal to numpy's int64 matmul."""
    rng = np.random.default_rng(10)
    for (M, N, K) in ((1, 1, 1), (17, 23, 31), (64, 3, 129), (5, 70, 8)):
        A = rng.integers(-4, 5, (M, K))
        B = rng.integers(-4, 5, (K, N))
        C0 = rng.integers(-4, 5, (M, N))
        want = (2 * (A @ B) - C0).astype(np.float64)
        for ta, tb in COMBOS:
            out, _ = _run(orc, A, B, ta, tb, 2.0, -1.0, C0, pad=(1, 0, 2))
            _exact(out, want, "int %s ta=%d tb=%d" % ((M, N, K), ta, tb))


def pin_library_float64(orc):
    """Random float data against torch.matmul in float64 on the CPU (a library routine)."""
    rng = np.random.default_rng(12)
    for (M, N, K) in ((33, 17, 65), (128, 96, 257), (3, 200, 511)):
        A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
        B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
        C0 = rng.uniform(-1, 1, (M, N)).astype(np.float32)
        want = (1.25 * torch.from_numpy(A).double() @ torch.from_numpy(B).double()
                - 0.5 * torch.from_numpy(C0).double()).numpy()
        for ta, tb in COMBOS:
            out, mag = _run(orc, A, B, ta, tb, 1.25, -0.5, C0, pad=(0, 3, 1))
            err = np.abs(out - want)
            assert np.all(err <= 1e-12 * mag), "float64 library %s ta=%d tb=%d: %g" % (
                (M, N, K), ta, tb, (err / mag).max())


def pin_batched(orc):
    """A strided batch equals the single problems one by one; stride 0 broadcasts."""
    rng = np.random.default_rng(13)
    batch, M, N, K = 3, 5, 4, 6
    for (ta, tb), broadcast_b in itertools.product(COMBOS, (False, True)):
        lda, ldb, ldc = (M if ta else K) + 1, (K if tb else N) + 2, N + 1
        sA, sC = lda * (K if ta else M) + 3, ldc * M + 5
        sB = 0 if broadcast_b else ldb * (N if tb else K) + 1
        A = rng.uniform(-1, 1, sA * batch).astype(np.float32)
        B = rng.uniform(-1, 1, ldb * (N if tb else K) + sB * batch).astype(np.float32)
        C0 = rng.uniform(-1, 1, sC * batch).astype(np.float32)
        out, mag = orc.gemm_strided_batched(ta, tb, M, N, K, 0.5, A, lda, sA, B, ldb, sB, 1.5,
                                            C0, ldc, sC, batch)
        for b in range(batch):
            o, m = orc.gemm(ta, tb, M, N, K, 0.5, A[b * sA:], lda, B[b * sB:], ldb, 1.5,
                            C0[b * sC:], ldc)
            _exact(out[b], o, "batch %d" % b)
            _exact(mag[b], m, "batch %d mag" % b)


def pin_fused_consistency(orc):
    """Fused = ReLU(unfused + bias[col]) and the bias is broadcast down the rows."""
    rng = np.random.default_rng(14)
    M, N, K = 8, 12, 20
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    b = rng.uniform(-1, 1, N).astype(np.float32)
    for ta, tb in COMBOS:
        plain, _ = _run(orc, A, B, ta, tb)
        biased, _ = _run(orc, A, B, ta, tb, bias=b)
        fused, _ = _run(orc, A, B, ta, tb, bias=b, relu=True)
        relu_only, _ = _run(orc, A, B, ta, tb, relu=True)
        _exact(biased, plain + b.astype(np.float64)[None, :], "bias broadcast")
        _exact(fused, np.maximum(biased, 0.0), "relu(bias)")
        _exact(relu_only, np.maximum(plain, 0.0), "relu only")
        assert (fused == 0).any() and (fused > 0).any()


def pin_row_bias_is_column_bias_of_the_transpose(orc):
    """A bias per row of C is a bias per column of C^T = B^T A^T (and ReLU commutes)."""
    rng = np.random.default_rng(17)
    M, N, K = 9, 7, 12
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    r = rng.uniform(-1, 1, M).astype(np.float32)
    for relu in (False, True):
        out, mag = orc.gemm(0, 0, M, N, K, 1.0, A.reshape(-1), K, B.reshape(-1), N, row_bias=r,
                            relu=relu)
        outT, magT = orc.gemm(1, 1, N, M, K, 1.0, B.reshape(-1), N, A.reshape(-1), K, bias=r,
                              relu=relu)
        _exact(outT, out.T, "row bias vs column bias of the transpose")
        _exact(magT, mag.T, "row bias mag")
        assert (out != _run(orc, A, B, 0, 0, relu=relu)[0]).any()


def pin_magnitude(orc):
    """mag(A, B, C0, b) equals the value computed on |A|, |B|, |C0|, |b|, |alpha|, |beta|."""
    rng = np.random.default_rng(15)
    M, N, K = 6, 9, 14
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    C0 = rng.uniform(-1, 1, (M, N)).astype(np.float32)
    b = rng.uniform(-1, 1, N).astype(np.float32)
    for ta, tb in COMBOS:
        _, mag = _run(orc, A, B, ta, tb, -1.5, -0.25, C0, b)
        absval, _ = _run(orc, np.abs(A), np.abs(B), ta, tb, 1.5, 0.25, np.abs(C0), np.abs(b))
        _exact(mag, absval, "mag ta=%d tb=%d" % (ta, tb))


def pin_row_subset_and_threads(orc):
    """Selected rows equal the same rows of the full result; thread count changes nothing."""
    rng = np.random.default_rng(16)
    M, N, K = 37, 19, 23
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    for ta, tb in COMBOS:
        full, fmag = _run(orc, A, B, ta, tb, threads=1)
        full4, _ = _run(orc, A, B, ta, tb, threads=4)
        _exact(full4, full, "threads")
        rows = np.array([36, 0, 5, 5, 17])
        sub, smag = _run(orc, A, B, ta, tb, rows=rows, threads=3)
        _exact(sub, full[rows], "rows")
        _exact(smag, fmag[rows], "rows mag")


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
