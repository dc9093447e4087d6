"""The six workloads at full size, launched exactly as bench.py launches them (through
fgemm_sgemm_staged with the model's staging choice, its default, and through the plain
entry points) and compared element by element with the FP64 oracle within 1e-5 * mag:
the whole output of the square problems (256^3, 1024^3 with alpha/beta, 4096^3), 4096
whole rows of the 8192-row fully-connected layer (every tile boundary included), and
two whole problems plus sampled rows of others for the batched QK^T and Score x V
(tests/workload_ref.py has the row choice)."""

import numpy as np
import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
from dense_fp32_gemm_sm_gb300 import workloads
from gpu_harness import REL_TOL
import workload_ref

pytestmark = pytest.mark.gpu


def run_workload(w, entry="plain"):
    dA, dB = w.A.cuda(), w.B.cuda()
    dbias = w.bias.cuda() if w.bias is not None else None
    nb = max(1, w.batch)
    dC = torch.empty((nb, w.M, w.N) if w.batch else (w.M, w.N), device="cuda")
    if w.C0 is not None:
        dC.copy_(w.C0)
    sA, sB, sC = (w.M * w.K, w.N * w.K, w.M * w.N) if w.batch else (0, 0, 0)
    if entry == "staged":
        need = fg.staged_workspace_size(w.ta, w.tb, w.M, w.N, w.K, nb)
        ws = torch.full((max(1, need // 4),), float("nan"), device="cuda")
        fg.sgemm_staged(w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, sA, dB, w.ldb, sB, w.beta,
                        dC, w.ldc, sC, nb, dbias, w.relu, fg.STAGE_AUTO, ws, need)
    elif w.batch:
        fg.sgemm_strided_batched(w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, w.M * w.K, dB,
                                 w.ldb, w.N * w.K, w.beta, dC, w.ldc, w.M * w.N, w.batch)
    elif w.bias is not None or w.relu:
        fg.sgemm_bias_relu(w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, dB, w.ldb, w.beta, dC,
                           w.ldc, dbias, w.relu)
    else:
        fg.sgemm(w.ta, w.tb, w.M, w.N, w.K, w.alpha, dA, w.lda, dB, w.ldb, w.beta, dC, w.ldc)
    torch.cuda.synchronize()
    return dC.cpu().numpy()


@pytest.mark.parametrize("entry", ["staged", "plain"])
@pytest.mark.parametrize("name", workloads.WORKLOADS)
def test_workload_against_oracle(name, entry):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    w = workload_ref.workload(name)
    C = run_workload(w, entry)
    workload_ref.compare(name, C, REL_TOL)
    if w.batch:
        assert workload_ref.checked_rows(name) >= 4096
    elif w.M <= 4096:
        assert workload_ref.checked_rows(name) == w.M  # the whole output
    else:
        assert workload_ref.checked_rows(name) >= 4096
    if w.relu:
        assert (C == 0).any() and (C > 0).any()


def test_fc_fused_equals_unfused_plus_epilogue():
    """The fused layer equals ReLU(plain GEMM + bias) computed from the library's own
    unfused result: the epilogue adds nothing but bias and ReLU (GEMM 优化详解, Level 6)."""
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    w = workload_ref.workload("fc8192x4096x11008")
    dA, dB, dbias = w.A.cuda(), w.B.cuda(), w.bias.cuda()
    fused = torch.empty((w.M, w.N), device="cuda")
    plain = torch.empty((w.M, w.N), device="cuda")
    fg.sgemm_bias_relu(w.ta, w.tb, w.M, w.N, w.K, 1.0, dA, w.lda, dB, w.ldb, 0.0, fused, w.ldc,
                       dbias, True)
    fg.sgemm(w.ta, w.tb, w.M, w.N, w.K, 1.0, dA, w.lda, dB, w.ldb, 0.0, plain, w.ldc)
    torch.cuda.synchronize()
    # same kernel configuration, same summation order: x + b rounds once, ReLU is exact
    expect = torch.clamp_min(plain + dbias, 0.0)
    assert torch.equal(fused, expect)


def test_bench_workloads_stage_as_measured():
    """On a 152-SM GB300 the model copies A k-major for 4096^3 and the FC layer, Q and K
    for QK^T, and nothing for the others: the staged legs above cover both paths."""
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms != 152:
        pytest.skip("expectations measured on 152 SMs")
    want = {"square256": 0, "square1024": 0, "square4096": 1, "fc8192x4096x11008": 1,
            "qkt128x2048x128": 3, "pv128x2048x2048x128": 0}
    for name in workloads.WORKLOADS:
        w = workload_ref.workload(name)
        got = fg.staged_choice(w.ta, w.tb, w.M, w.N, w.K, max(1, w.batch), False, False, True,
                               True, sms)
        assert got == want[name], name
