"""Failure detection of the tensor-core kernel without a GPU fault.

A test-only hook makes the TMA producer withhold one k-block, as if its copy never
arrived.  The consumers' bounded waits then run out after a short limit; the kernel
records FGEMM_ERR_TIMEOUT, drains its own copies and MMAs, frees its tensor memory
and returns.  The host reads the status, and the same context then computes the
next GEMM exactly.
"""

import time

import numpy as np
import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
import oracle

pytestmark = pytest.mark.gpu

LIMIT_NS = 200_000_000  # 0.2 s per wait


def _operands(ta, tb, M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    A = torch.randint(-4, 5, (K, M) if ta else (M, K), generator=g).float()
    B = torch.randint(-4, 5, (N, K) if tb else (K, N), generator=g).float()
    return A, B


def _call(math, ta, tb, M, N, K, A, B, C):
    fg.gemm_math(math, ta, tb, M, N, K, 1.0, A, A.shape[1], 0, B, B.shape[1], 0, 0.0, C, N, 0, 1)


@pytest.mark.parametrize("math,ta,tb", [(fg.MATH_TF32, 0, 1), (fg.MATH_3XTF32, 0, 1),
                                        (fg.MATH_3XTF32, 0, 0), (fg.MATH_TF32, 1, 0)])
def test_withheld_copy_times_out_and_context_survives(math, ta, tb):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    M, N, K = 256, 256, 320  # 4 tiles, 10 k-blocks of 32
    A, B = _operands(ta, tb, M, N, K, seed=ta * 2 + tb)
    dA, dB = A.cuda(), B.cuda()
    C = torch.zeros(M, N, device="cuda")
    torch.cuda.synchronize()
    fg.device_status(clear=True)
    try:
        fg.debug_withhold_tensor_core(3, LIMIT_NS)
        t0 = time.perf_counter()
        _call(math, ta, tb, M, N, K, dA, dB, C)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        fg.debug_withhold_tensor_core(-1)
    assert fg.device_status(clear=True) == fg.ERR_TIMEOUT
    assert elapsed < 5.0, "the bounded waits took %.2f s" % elapsed
    assert fg.device_status(clear=False) == fg.OK  # cleared

    # The context is intact: the same call now gives the exact result.
    C.fill_(float("nan"))
    _call(math, ta, tb, M, N, K, dA, dB, C)
    torch.cuda.synchronize()
    assert fg.device_status() == fg.OK
    want, _ = oracle.gemm(ta, tb, M, N, K, 1.0, A.numpy().reshape(-1), A.shape[1],
                          B.numpy().reshape(-1), B.shape[1], want_mag=False)
    assert np.array_equal(C.cpu().numpy().astype(np.float64), want)


def test_cuda_core_kernel_unaffected_by_the_hook():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    M, N, K = 130, 70, 64
    A, B = _operands(0, 0, M, N, K, seed=9)
    C = torch.zeros(M, N, device="cuda")
    try:
        fg.debug_withhold_tensor_core(0, LIMIT_NS)
        fg.sgemm(0, 0, M, N, K, 1.0, A.cuda(), K, B.cuda(), N, 0.0, C, N)
        torch.cuda.synchronize()
    finally:
        fg.debug_withhold_tensor_core(-1)
    assert fg.device_status() == fg.OK
    want, _ = oracle.gemm(0, 0, M, N, K, 1.0, A.numpy().reshape(-1), K, B.numpy().reshape(-1), N,
                          want_mag=False)
    assert np.array_equal(C.cpu().numpy().astype(np.float64), want)
