"""The tcgen05 tensor-core path (TF32 and 3xTF32) against the FP64 oracle, in all
four transpose combinations (K-major operands go straight from TMA to the tensor
cores, MN-major ones are transposed on chip).

Small-integer data is exact in TF32 (hi = x, lo = 0), so both modes must be
bit-exact on it, like the CUDA-core kernel.  On uniform data TF32 must stay within
the method's TF32 bound 2e-3 * sum_k |a_ik||b_kj| (extended by |beta c| + |bias|),
and 3xTF32 within the FP32 bound 1e-5 * mag.
"""

import itertools

import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
from gpu_harness import Case, check

pytestmark = pytest.mark.gpu

TF32_TOL = 2e-3
MODES = [fg.MATH_TF32, fg.MATH_3XTF32]
SHAPES = [(128, 128, 32), (300, 200, 130), (257, 31, 515), (1, 1, 1), (129, 257, 33),
          (640, 384, 1024)]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    fg.library()
    fg.device_status(clear=True)


COMBOS = list(itertools.product((0, 1), (0, 1)))


@pytest.mark.parametrize("math", MODES, ids=["tf32", "3xtf32"])
@pytest.mark.parametrize("ta,tb", COMBOS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_integer_exact(math, ta, tb, shape):
    M, N, K = shape
    check(Case(ta=ta, tb=tb, M=M, N=N, K=K, alpha=2.0, beta=-0.5, math=math, pad=(4, 8, 4),
               seed=M * 7 + N + K))


@pytest.mark.parametrize("math", MODES, ids=["tf32", "3xtf32"])
@pytest.mark.parametrize("bias,relu", [(False, False), (True, False), (False, True), (True, True)])
def test_epilogue_options(math, bias, relu):
    for ta, tb in COMBOS:
        check(Case(ta=ta, tb=tb, M=200, N=152, K=96, bias=bias, relu=relu, beta=1.0, math=math,
                   seed=3))


@pytest.mark.parametrize("math", MODES, ids=["tf32", "3xtf32"])
@pytest.mark.parametrize("ta,tb", COMBOS)
def test_batched(math, ta, tb):
    check(Case(ta=ta, tb=tb, M=130, N=70, K=45, alpha=0.5, beta=1.0, batch=3, math=math, seed=5))


@pytest.mark.parametrize("ta,tb", COMBOS)
def test_uniform_tf32_within_tf32_bound(ta, tb):
    check(Case(ta=ta, tb=tb, M=515, N=387, K=1029, alpha=1.5, beta=0.5, ints=False,
               math=fg.MATH_TF32, seed=8), rel_tol=TF32_TOL)


@pytest.mark.parametrize("ta,tb", COMBOS)
def test_uniform_3xtf32_within_fp32_bound(ta, tb):
    worst = check(Case(ta=ta, tb=tb, M=515, N=387, K=1029, alpha=1.5, beta=0.5, ints=False,
                       math=fg.MATH_3XTF32, seed=9))
    assert worst < 1e-5


def test_tf32_is_not_fp32():
    # TF32 really drops mantissa bits: on uniform data its error is far above FP32's.
    worst = check(Case(ta=0, tb=1, M=256, N=256, K=512, ints=False, math=fg.MATH_TF32, seed=10),
                  rel_tol=TF32_TOL)
    assert worst > 1e-5


@pytest.mark.parametrize("math", MODES, ids=["tf32", "3xtf32"])
@pytest.mark.parametrize("ta,tb", COMBOS)
def test_unaligned_falls_back_to_fp32(math, ta, tb):
    # Calls the tensor-core kernel cannot take run the FP32 kernel: exact on integers and
    # within the FP32 bound on floats.
    check(Case(ta=ta, tb=tb, M=100, N=60, K=50, math=math, offset=(1, 0, 0), align_ld=False,
               seed=13, expect_tc=False))
    check(Case(ta=ta, tb=tb, M=100, N=60, K=50, math=math, offset=(0, 0, 0), pad=(1, 3, 0),
               align_ld=False, ints=False, seed=14, expect_tc=False))


@pytest.mark.parametrize("math", MODES, ids=["tf32", "3xtf32"])
def test_k_zero_and_alpha_zero(math):
    check(Case(ta=0, tb=1, M=70, N=90, K=0, alpha=3.0, beta=-2.0, bias=True, relu=True, math=math,
               expect_tc=False))
    check(Case(ta=0, tb=0, M=70, N=90, K=33, alpha=0.0, beta=0.5, a_nan=True, math=math,
               expect_tc=False))


def test_fp32_math_is_the_cuda_core_kernel():
    check(Case(ta=0, tb=1, M=190, N=100, K=64, math=fg.MATH_FP32, seed=14))
    check(Case(ta=0, tb=0, M=190, N=100, K=64, math=fg.MATH_FP32, ints=False, seed=15))


def test_bad_math_value():
    A = torch.zeros(16, device="cuda")
    st = fg.gemm_math(7, 0, 1, 4, 4, 4, 1.0, A, 4, 0, A, 4, 0, 0.0, A, 4, 0, 1, check=False)
    assert st == fg.ERR_INVALID_VALUE


def test_device_status_clean():
    torch.cuda.synchronize()
    assert fg.device_status(clear=False) == fg.OK


@pytest.mark.parametrize("math", MODES, ids=["tf32", "3xtf32"])
@pytest.mark.parametrize("ta,tb", COMBOS)
@pytest.mark.parametrize("shape", [(300, 200, 130), (257, 31, 515), (129, 257, 33), (520, 600, 96),
                                   (64, 36, 40)],
                         ids=lambda s: "x".join(map(str, s)))
def test_beta_zero_epilogue(math, ta, tb, shape):
    # beta = 0 with an aligned C and N a multiple of 4 takes the epilogue that stages
    # tiles in shared memory and writes them with TMA stores (clipped at the edges;
    # transposed tiles in NN); other N store directly.  C starts as NaN (any read of it
    # would show) and its padding columns hold a sentinel that must survive.
    M, N, K = shape
    check(Case(ta=ta, tb=tb, M=M, N=N, K=K, alpha=1.5, beta=0.0, bias=True, relu=True,
               c_nan=True, pad=(4, 8, 4), math=math, seed=M + 3 * N + K))
    check(Case(ta=ta, tb=tb, M=M, N=N, K=K, alpha=1.0, beta=0.0, c_nan=True, pad=(0, 0, 8),
               math=math, ints=False, seed=M + N),
          rel_tol=TF32_TOL if math == fg.MATH_TF32 else 1e-5)


@pytest.mark.parametrize("math", MODES, ids=["tf32", "3xtf32"])
@pytest.mark.parametrize("ta,tb", COMBOS)
@pytest.mark.parametrize("shape", [(2560, 2048, 64), (2048, 2560, 40)],
                         ids=lambda s: "x".join(map(str, s)))
def test_last_wave_split_into_half_tiles(math, ta, tb, shape):
    # 160 tiles of 128 x 256 (or 256 x 128) on a ~150-SM GPU: the last partial wave runs
    # as half tiles of 128 x 128.  Exact on integer data, every element checked.
    M, N, K = shape
    check(Case(ta=ta, tb=tb, M=M, N=N, K=K, alpha=1.0, beta=0.0, math=math, seed=M + N + K))
    check(Case(ta=ta, tb=tb, M=M, N=N, K=K, alpha=0.5, beta=1.0, bias=True, relu=True, math=math,
               pad=(4, 0, 4), seed=K))
