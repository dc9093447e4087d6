"""fgemm_sgemm_splitk_noalloc: the split-K GEMM for callers that may not allocate
device memory (a plugin inside a program that owns all GPU memory, a
latency-critical loop that cannot pay for cudaMalloc, a fixed memory budget).

The entry point keeps its partial products in the library's fixed device array
instead of a caller workspace.  It must give the same result as
fgemm_sgemm_splitk with a workspace, on two calls in a row with different data
(the array keeps the previous call's contents, which must not leak into the next
result), and reject problems that do not fit the array.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test.
"""

import numpy as np
import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
import oracle
from dense_fp32_gemm_sm_gb300 import workloads

pytestmark = pytest.mark.gpu

REL_TOL = 1e-5
FLT_MIN = float(np.finfo(np.float32).tiny)


def _problem(seed, M, N, K, ta, tb):
    g = workloads.generator(seed)
    A = workloads.uniform(g, (K, M) if ta else (M, K))
    B = workloads.uniform(g, (N, K) if tb else (K, N))
    C0 = workloads.uniform(g, (M, N))
    bias = workloads.uniform(g, (N,))
    return A, B, C0, bias


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")
def test_noalloc_matches_workspace_entry_point_on_two_calls():
    # Two different problems back to back through the same fixed array.
    for seed, (M, N, K, ta, tb, splits, relu) in enumerate(
            [(1024, 1024, 1024, 0, 0, 4, False), (300, 500, 2000, 1, 1, 3, True)]):
        A, B, C0, bias = _problem(seed + 40, M, N, K, ta, tb)
        assert fg.splitk_workspace_size(M, N, K, splits) <= fg.NOALLOC_SCRATCH_BYTES
        dA, dB, dbias = A.cuda(), B.cuda(), bias.cuda()
        lda, ldb = A.shape[1], B.shape[1]

        ref = C0.cuda()
        need = fg.splitk_workspace_size(M, N, K, splits)
        ws = torch.empty(need // 4, device="cuda")
        fg.sgemm_splitk(ta, tb, M, N, K, 1.5, dA, lda, dB, ldb, 0.5, ref, N, dbias, relu, splits,
                        ws, need)

        out = C0.cuda()
        fg.sgemm_splitk_noalloc(ta, tb, M, N, K, 1.5, dA, lda, dB, ldb, 0.5, out, N, dbias, relu,
                                splits)
        torch.cuda.synchronize()

        got, want = out.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)
        # within the tolerance of the parity tests, relative to the oracle's magnitudes
        rows = np.arange(0, M, max(1, M // 64))
        _, mag = oracle.gemm(ta, tb, M, N, K, 1.5, A.numpy().reshape(-1), lda,
                             B.numpy().reshape(-1), ldb, 0.5, C0.numpy().reshape(-1), N,
                             bias=bias.numpy(), relu=relu, rows=rows)
        assert (np.abs(got[rows] - want[rows]) <= REL_TOL * mag + FLT_MIN).all()
        # the same kernels in the same order: the same bits
        assert np.array_equal(got, want)


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")
def test_noalloc_rejects_problems_larger_than_the_array():
    M = N = 2048
    K, splits = 4096, 4  # 4 x 2048 x 2048 floats = 64 MiB of partial products
    assert fg.splitk_workspace_size(M, N, K, splits) > fg.NOALLOC_SCRATCH_BYTES
    A = torch.zeros(M * K, device="cuda")
    B = torch.zeros(K * N, device="cuda")
    C = torch.full((M, N), 7.0, device="cuda")
    st = fg.sgemm_splitk_noalloc(0, 0, M, N, K, 1.0, A, K, B, N, 0.0, C, N, None, False, splits,
                                 check=False)
    torch.cuda.synchronize()
    assert st == fg.ERR_NOT_SUPPORTED
    assert bool((C == 7.0).all())  # nothing ran
