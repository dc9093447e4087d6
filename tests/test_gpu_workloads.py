"""The five workloads at full size, launched exactly as bench.py launches them,
checked on sampled output rows (all columns of each sampled row) against the
FP64 oracle within 1e-5 * mag.  Sampled rows include the first and last row
and both sides of CTA-tile boundaries."""

import numpy as np
import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
import oracle
from dense_fp32_gemm_sm_gb300 import workloads
from gpu_harness import FLT_MIN, REL_TOL

pytestmark = pytest.mark.gpu


def sample_rows(M, n, seed):
    rng = np.random.default_rng(seed)
    edges = [0, 1, 63, 64, 127, 128, M // 2, M - 129, M - 128, M - 2, M - 1]
    extra = rng.choice(M, size=max(0, n - len(edges)), replace=False)
    return np.unique(np.clip(np.concatenate([edges, extra]), 0, M - 1)).astype(np.int64)


def run_workload(w):
    dA, dB = w.A.cuda(), w.B.cuda()
    dbias = w.bias.cuda() if w.bias is not None else None
    nb = max(1, w.batch)
    dC = torch.empty((nb, w.M, w.N) if w.batch else (w.M, w.N), device="cuda")
    if w.C0 is not None:
        dC.copy_(w.C0)
    if w.batch:
        fg.sgemm_strided_batched(w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, w.M * w.K, dB,
                                 w.ldb, w.N * w.K, w.beta, dC, w.ldc, w.M * w.N, w.batch)
    elif w.bias is not None or w.relu:
        fg.sgemm_bias_relu(w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, dB, w.ldb, w.beta, dC,
                           w.ldc, dbias, w.relu)
    else:
        fg.sgemm(w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, dB, w.ldb, w.beta, dC, w.ldc)
    torch.cuda.synchronize()
    return dC.cpu().numpy()


def compare(got_rows, want, mag):
    err = np.abs(got_rows.astype(np.float64) - want)
    bound = REL_TOL * mag + FLT_MIN
    assert not np.isnan(got_rows).any()
    assert (err <= bound).all(), "worst err/bound %g" % (err / bound).max()


@pytest.mark.parametrize("name", workloads.WORKLOADS[:4])
def test_single_workload_sampled(name):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    w = workloads.make(name)
    C = run_workload(w)
    rows = sample_rows(w.M, 48 if w.M >= 4096 else w.M, seed=len(name))
    C0 = w.C0.numpy().reshape(-1) if w.C0 is not None else None
    want, mag = oracle.gemm(w.ta, w.tb, w.M, w.N, w.K, w.alpha, w.A.numpy().reshape(-1), w.lda,
                            w.B.numpy().reshape(-1), w.ldb, w.beta, C0, w.ldc,
                            bias=w.bias, relu=w.relu, rows=rows)
    compare(C[rows], want, mag)
    if w.relu:
        assert (C[rows] == 0).any() and (C[rows] > 0).any()


@pytest.mark.parametrize("name", ["qkt128x2048x128", "pv128x2048x2048x128"])
def test_batched_attention_sampled(name):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    w = workloads.make(name)
    C = run_workload(w)
    A, B = w.A.numpy(), w.B.numpy()
    for b in (0, 1, 63, 127):
        rows = sample_rows(w.M, 24, seed=b)
        want, mag = oracle.gemm(w.ta, w.tb, w.M, w.N, w.K, w.alpha, A[b].reshape(-1), w.lda,
                                B[b].reshape(-1), w.ldb, rows=rows)
        compare(C[b][rows], want, mag)
