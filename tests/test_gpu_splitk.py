"""Split-K GEMM (fgemm_sgemm_splitk) against the FP64 oracle.

The K range is cut into slices computed as separate GEMMs into a workspace and
summed in a fixed order: on small-integer data the result is exact for every
number of slices, on uniform data within 1e-5 * mag, and two calls agree bit for bit.
"""

import itertools

import numpy as np
import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
import oracle
from dense_fp32_gemm_sm_gb300 import workloads
from gpu_harness import FLT_MIN, REL_TOL

pytestmark = pytest.mark.gpu

COMBOS = list(itertools.product((0, 1), (0, 1)))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    fg.library()


def run_case(ta, tb, M, N, K, splits, alpha=1.0, beta=0.0, bias=False, relu=False, ints=True,
             seed=0):
    g = workloads.generator(seed)
    draw = (lambda shape: workloads.small_ints(g, shape)) if ints else (
        lambda shape: workloads.uniform(g, shape))
    A = draw((K, M) if ta else (M, K))
    B = draw((N, K) if tb else (K, N))
    C0 = workloads.small_ints(g, (M, N))
    b = workloads.small_ints(g, (N,)) if bias else None
    lda, ldb = A.shape[1], B.shape[1]
    dC = C0.cuda()
    need = fg.splitk_workspace_size(M, N, K, splits)
    ws = torch.full((max(need // 4, 1),), float("nan"), device="cuda")
    fg.sgemm_splitk(ta, tb, M, N, K, alpha, A.cuda(), lda, B.cuda(), ldb, beta, dC, N,
                    b.cuda() if b is not None else None, relu, splits, ws, need)
    torch.cuda.synchronize()
    want, mag = oracle.gemm(ta, tb, M, N, K, alpha, A.numpy().reshape(-1), lda,
                            B.numpy().reshape(-1), ldb, beta, C0.numpy().reshape(-1), N,
                            bias=None if b is None else b.numpy(), relu=relu)
    return dC.cpu().numpy().astype(np.float64), want, mag


@pytest.mark.parametrize("ta,tb", COMBOS)
@pytest.mark.parametrize("splits", [1, 2, 3, 4, 7, 16])
def test_integer_exact(ta, tb, splits):
    for (M, N, K) in ((256, 256, 256), (300, 200, 1000), (64, 96, 4099)):
        got, want, _ = run_case(ta, tb, M, N, K, splits, alpha=2.0, beta=-0.5, seed=splits)
        assert np.array_equal(got, want), (M, N, K, splits)


@pytest.mark.parametrize("bias,relu", [(True, True), (True, False), (False, True)])
def test_epilogue(bias, relu):
    got, want, _ = run_case(0, 0, 130, 70, 520, 4, beta=1.0, bias=bias, relu=relu, seed=3)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("ta,tb", COMBOS)
def test_uniform_within_bound(ta, tb):
    got, want, mag = run_case(ta, tb, 257, 129, 3000, 5, alpha=1.5, beta=0.5, ints=False, seed=4)
    assert (np.abs(got - want) <= REL_TOL * mag + FLT_MIN).all()


def test_deterministic():
    g = workloads.generator(7)
    M, N, K = 512, 384, 2048
    A, B = workloads.uniform(g, (M, K)).cuda(), workloads.uniform(g, (K, N)).cuda()
    need = fg.splitk_workspace_size(M, N, K, 8)
    ws = torch.empty(need // 4, device="cuda")
    outs = []
    for _ in range(2):
        C = torch.empty(M, N, device="cuda")
        fg.sgemm_splitk(0, 0, M, N, K, 1.0, A, K, B, N, 0.0, C, N, None, False, 8, ws, need)
        outs.append(C)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


def test_full_size_square1024_sampled():
    w = workloads.make("square1024")
    need = fg.splitk_workspace_size(w.M, w.N, w.K, 4)
    ws = torch.empty(need // 4, device="cuda")
    C = w.C0.cuda()
    fg.sgemm_splitk(0, 0, w.M, w.N, w.K, w.alpha, w.A.cuda(), w.lda, w.B.cuda(), w.ldb, w.beta, C,
                    w.ldc, None, False, 4, ws, need)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 127, 128, 511, 512, 1022, 1023])
    want, mag = oracle.gemm(0, 0, w.M, w.N, w.K, w.alpha, w.A.numpy().reshape(-1), w.lda,
                            w.B.numpy().reshape(-1), w.ldb, w.beta, w.C0.numpy().reshape(-1), w.ldc,
                            rows=rows)
    got = C.cpu().numpy()[rows].astype(np.float64)
    assert (np.abs(got - want) <= REL_TOL * mag + FLT_MIN).all()
