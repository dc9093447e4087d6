"""The tensor-core path on the full-size workloads, launched as bench.py --math
launches them, checked on sampled output rows against the FP64 oracle: TF32 within
2e-3 * mag, 3xTF32 within the FP32 bound 1e-5 * mag.  Sampled rows include both
sides of the 128- and 256-row tile boundaries and the last rows."""

import numpy as np
import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
import oracle
from dense_fp32_gemm_sm_gb300 import workloads
from gpu_harness import FLT_MIN

pytestmark = pytest.mark.gpu

TOL = {fg.MATH_TF32: 2e-3, fg.MATH_3XTF32: 1e-5}


def sample_rows(M, n, seed):
    rng = np.random.default_rng(seed)
    edges = [0, 1, 127, 128, 255, 256, 257, M // 2, M - 257, M - 256, M - 129, M - 128, M - 1]
    extra = rng.choice(M, size=max(0, n - len(edges)), replace=False)
    return np.unique(np.clip(np.concatenate([edges, extra]), 0, M - 1)).astype(np.int64)


def run(w, math):
    nb = max(1, w.batch)
    dA, dB = w.A.cuda(), w.B.cuda()
    dbias = w.bias.cuda() if w.bias is not None else None
    dC = torch.empty((nb, w.M, w.N) if w.batch else (w.M, w.N), device="cuda")
    if w.C0 is not None:
        dC.copy_(w.C0)
    sA = w.M * w.K if w.batch else 0
    sB = w.N * w.K if w.batch else 0
    sC = w.M * w.N if w.batch else 0
    fg.gemm_math(math, w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, sA, dB, w.ldb, sB, w.beta,
                 dC, w.ldc, sC, nb, dbias, w.relu)
    torch.cuda.synchronize()
    assert fg.device_status() == fg.OK
    return dC.cpu().numpy()


def compare(got, want, mag, tol):
    assert not np.isnan(got).any()
    err = np.abs(got.astype(np.float64) - want)
    bound = tol * mag + FLT_MIN
    assert (err <= bound).all(), "worst err/bound %g" % (err / bound).max()


@pytest.mark.parametrize("math", [fg.MATH_TF32, fg.MATH_3XTF32], ids=["tf32", "3xtf32"])
@pytest.mark.parametrize("name", workloads.WORKLOADS)
def test_workload_sampled(name, math):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    w = workloads.make(name)
    C = run(w, math)
    if w.batch:
        A, B = w.A.numpy(), w.B.numpy()
        for b in (0, 77, 127):
            rows = sample_rows(w.M, 20, seed=b)
            want, mag = oracle.gemm(w.ta, w.tb, w.M, w.N, w.K, w.alpha, A[b].reshape(-1), w.lda,
                                    B[b].reshape(-1), w.ldb, rows=rows)
            compare(C[b][rows], want, mag, TOL[math])
        return
    rows = sample_rows(w.M, 32 if w.M >= 4096 else w.M, seed=len(name))
    C0 = w.C0.numpy().reshape(-1) if w.C0 is not None else None
    want, mag = oracle.gemm(w.ta, w.tb, w.M, w.N, w.K, w.alpha, w.A.numpy().reshape(-1), w.lda,
                            w.B.numpy().reshape(-1), w.ldb, w.beta, C0, w.ldc, bias=w.bias,
                            relu=w.relu, rows=rows)
    compare(C[rows], want, mag, TOL[math])
