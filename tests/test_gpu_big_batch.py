"""Batches of more than 65535 problems (the limit of one grid dimension).

The per-problem grid runs such a batch in chunks of 65535 launches' worth of
problems, the last-wave splits walk one linear tile order over all problems, the
staged call's copy kernel splits its batch the same way, and the persistent tensor-core
kernel walks the tiles of all problems as one list of work items.  Small-integer data, so every
result is exact: the problems on both sides of each chunk boundary, the first and the
last are compared with the FP64 oracle element by element, and every problem is
compared with a float64 CPU matmul of the same integers (exact as well).
"""

import numpy as np
import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
import oracle
from dense_fp32_gemm_sm_gb300 import workloads

pytestmark = pytest.mark.gpu

BATCH = 65535 + 65535 // 2 + 7  # two chunks and a ragged third
M, N, K = 8, 12, 20
CHECKED = sorted({0, 1, 65533, 65534, 65535, 65536, 65537, 2 * 65535 - 1, 2 * 65535,
                  BATCH - 2, BATCH - 1} & set(range(BATCH)))


def _config(name):
    ids = [i for i in range(fg.num_configs()) if fg.config_name(i) == name]
    assert len(ids) == 1
    return ids[0]


@pytest.fixture(scope="module")
def operands():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    fg.library()
    g = workloads.generator(200)
    A = workloads.small_ints(g, (BATCH, M, K))   # op(A) = N: stored M x K
    Bt = workloads.small_ints(g, (BATCH, N, K))  # op(B) = T: stored N x K
    want = torch.bmm(A.double(), Bt.double().transpose(1, 2))
    return A, Bt, want


def _check(C, A, Bt, want, alpha):
    got = C.cpu()
    assert torch.equal(got.double(), alpha * want), "some problem differs from the CPU matmul"
    for b in CHECKED:
        o, _ = oracle.gemm(0, 1, M, N, K, alpha, A[b].numpy().reshape(-1), K,
                           Bt[b].numpy().reshape(-1), K)
        assert np.array_equal(got[b].numpy().astype(np.float64), o), "problem %d" % b


@pytest.mark.parametrize("config", [None, "simt_32x32x16_t4x4_s4", "simt_128x128_t8x8_kchain"])
def test_plain_batch_beyond_one_grid_dimension(operands, config):
    A, Bt, want = operands
    dA, dB = A.cuda(), Bt.cuda()
    C = torch.full((BATCH, M, N), float("nan"), device="cuda")
    cfg = -1 if config is None else _config(config)
    fg.gemm_explicit(cfg, 0, 1, M, N, K, 2.0, dA, K, M * K, dB, K, N * K, 0.0, C, N, M * N, BATCH)
    torch.cuda.synchronize()
    _check(C, A, Bt, want, 2.0)


def test_staged_batch_beyond_one_grid_dimension(operands):
    """Both operands transposed by the copy kernel in chunks of 65535 problems."""
    A, Bt, want = operands
    dA, dB = A.cuda(), Bt.cuda()
    C = torch.full((BATCH, M, N), float("nan"), device="cuda")
    need = fg.staged_workspace_size(0, 1, M, N, K, BATCH)
    ws = torch.full((need // 4,), float("nan"), device="cuda")
    # both operands copied k-major (two copy launches of three chunks each)
    fg.sgemm_staged(0, 1, M, N, K, -0.5, dA, K, M * K, dB, K, N * K, 0.0, C, N, M * N, BATCH,
                    None, False, 3, ws, need)
    torch.cuda.synchronize()
    _check(C, A, Bt, want, -0.5)


def test_repitched_batch_beyond_one_grid_dimension(operands):
    """Both operands already k-major (op(A) = T, op(B) = N) and copied row by row into
    aligned rows, in chunks of 65535 problems."""
    A, Bt, want = operands
    At = A.transpose(1, 2).contiguous()  # K x M: op(A) = T
    Bk = Bt.transpose(1, 2).contiguous()  # K x N: op(B) = N
    dA, dB = At.cuda(), Bk.cuda()
    C = torch.full((BATCH, M, N), float("nan"), device="cuda")
    need = fg.staged_workspace_size(1, 0, M, N, K, BATCH)
    ws = torch.full((need // 4,), float("nan"), device="cuda")
    fg.sgemm_staged(1, 0, M, N, K, 1.0, dA, M, M * K, dB, N, N * K, 0.0, C, N, M * N, BATCH,
                    None, False, 3, ws, need)
    torch.cuda.synchronize()
    _check(C, A, Bt, want, 1.0)


@pytest.mark.parametrize("math", [fg.MATH_TF32, fg.MATH_3XTF32], ids=["tf32", "3xtf32"])
def test_tensor_core_batch_beyond_one_grid_dimension(operands, math):
    """The persistent tensor-core kernel walks (problem, tile) items of all 98309 problems
    (the batch is the tensor maps' third dimension)."""
    A, Bt, want = operands
    dA, dB = A.cuda(), Bt.cuda()
    C = torch.full((BATCH, M, N), float("nan"), device="cuda")
    assert fg.math_supported(math, 0, 1, M, N, K, 0.5, dA, K, M * K, dB, K, N * K, BATCH) == 1
    fg.gemm_math(math, 0, 1, M, N, K, 0.5, dA, K, M * K, dB, K, N * K, 0.0, C, N, M * N, BATCH)
    torch.cuda.synchronize()
    assert fg.device_status() == fg.OK
    _check(C, A, Bt, want, 0.5)
