"""The tensor-core path on the six full-size workloads, launched as bench.py --math
launches them, compared element by element with the FP64 oracle on the rows of
tests/workload_ref.py (the whole output of the square problems, 4096 rows of the
layer, two whole problems plus samples of the batches): TF32 within 2e-3 * mag,
3xTF32 within the FP32 bound 1e-5 * mag.  Every call is first confirmed to run on
the tensor cores (fgemm_math_supported)."""

import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
from dense_fp32_gemm_sm_gb300 import workloads
import workload_ref

pytestmark = pytest.mark.gpu

TOL = {fg.MATH_TF32: 2e-3, fg.MATH_3XTF32: 1e-5}


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
    assert fg.math_supported(math, w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, sA, dB, w.ldb,
                             sB, nb) == 1, "the tensor-core kernel would not run this workload"
    fg.gemm_math(math, w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, sA, dB, w.ldb, sB, w.beta,
                 dC, w.ldc, sC, nb, dbias, w.relu)
    torch.cuda.synchronize()
    assert fg.device_status() == fg.OK
    return dC.cpu().numpy()


@pytest.mark.parametrize("math", [fg.MATH_TF32, fg.MATH_3XTF32], ids=["tf32", "3xtf32"])
@pytest.mark.parametrize("name", workloads.WORKLOADS)
def test_workload_against_oracle(name, math):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    w = workload_ref.workload(name)
    C = run(w, math)
    workload_ref.compare(name, C, TOL[math])
