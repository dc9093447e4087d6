"""fgemm_gemm_math_staged against the FP64 oracle.

The call copies operands K-major into a caller workspace (transposed when MN-major,
into aligned rows when K-major but not 16-byte aligned) and runs the tensor-core kernel
on the copies.  Checked here, through the C ABI: every layout with every copy mask and
the library's own choice, in TF32 and 3xTF32, on ragged sizes over several tiles
(integer data: bit-exact); uniform data within each arithmetic's bound; strided batches
with and without a shared operand; unaligned operands, which the plain tensor-core call
hands to the CUDA cores and the staged call runs on the tensor cores (its error is then
TF32's, far above FP32 rounding); alpha = 0 and K = 0 (no copies); FGEMM_MATH_FP32, which
is fgemm_sgemm_staged.  The harness fills the workspace with NaN, so an element read
before a copy wrote it would show.
"""

import itertools

import numpy as np
import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
from gpu_harness import Case, check, run

pytestmark = pytest.mark.gpu

COMBOS = list(itertools.product((0, 1), (0, 1)))
MODES = [fg.MATH_TF32, fg.MATH_3XTF32]
IDS = ["tf32", "3xtf32"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    fg.library()


@pytest.mark.parametrize("stage", [fg.STAGE_AUTO, 0, 1, 2, 3])
@pytest.mark.parametrize("ta,tb", COMBOS)
@pytest.mark.parametrize("math", MODES, ids=IDS)
def test_every_layout_and_mask_integer_exact(math, ta, tb, stage):
    check(Case(ta=ta, tb=tb, M=300, N=260, K=333, alpha=1.5, beta=0.5, bias=True, relu=True,
               pad=(4, 8, 4), math=math, stage=stage, expect_tc=None,
               seed=700 + 10 * (stage + 1) + 2 * ta + tb))


@pytest.mark.parametrize("ta,tb", COMBOS)
@pytest.mark.parametrize("math", MODES, ids=IDS)
def test_uniform_within_the_bound(math, ta, tb):
    # 1700 x 1650 x 300: 128 x 256 / 128 x 128 tiles and a last partial wave
    check(Case(ta=ta, tb=tb, M=1700, N=1650, K=300, alpha=-0.75, beta=1.25, ints=False,
               bias=True, math=math, stage=fg.STAGE_AUTO, expect_tc=None, seed=720 + 2 * ta + tb),
          rel_tol=2e-3 if math == fg.MATH_TF32 else 1e-5)


@pytest.mark.parametrize("share", [(False, False), (True, False), (False, True)])
@pytest.mark.parametrize("math", MODES, ids=IDS)
def test_strided_batch_and_shared_operands(math, share):
    check(Case(ta=1, tb=0, M=200, N=176, K=96, alpha=1.0, beta=-1.0, batch=5, math=math,
               stage=3, share_a=share[0], share_b=share[1], expect_tc=None,
               seed=730 + 7 * share[0] + share[1]))


@pytest.mark.parametrize("ta,tb", COMBOS)
def test_unaligned_operands_run_on_the_tensor_cores(ta, tb):
    # odd leading dimensions and pointers 4 bytes past a 16-byte boundary: the plain
    # tensor-core call falls back to the CUDA cores (FP32 error, about 1e-7 of the
    # magnitude); after the copies the call runs on the tensor cores (TF32 error)
    M, N, K = 333, 222, 111
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert fg.math_staged_choice(fg.MATH_TF32, ta, tb, M, N, K, 1, 0, 0, 0, 0, sms) == 3
    base = dict(ta=ta, tb=tb, M=M, N=N, K=K, alpha=2.0, beta=0.0, ints=False, align_ld=False,
                pad=(1, 3, 1), offset=(1, 3, 2), math=fg.MATH_TF32, seed=740 + 2 * ta + tb)
    got, want, mag, ok = run(Case(**base, stage=fg.STAGE_AUTO, expect_tc=None))
    assert ok
    err = np.abs(got.astype(np.float64) - want) / (mag + 1e-30)
    assert err.max() <= 2e-3, "outside the TF32 bound"
    assert err.max() > 1e-5, "FP32 accuracy: the call did not run on the tensor cores"
    got0, _, _, _ = run(Case(**base, expect_tc=False))  # the plain call: CUDA cores
    err0 = np.abs(got0.astype(np.float64) - want) / (mag + 1e-30)
    assert err0.max() <= 1e-5


@pytest.mark.parametrize("math", MODES, ids=IDS)
def test_no_products_copy_nothing(math):
    check(Case(ta=1, tb=0, M=129, N=131, K=64, alpha=0.0, beta=0.5, a_nan=True, bias=True,
               math=math, stage=3, expect_tc=None, seed=750))
    check(Case(ta=1, tb=0, M=129, N=131, K=0, alpha=1.0, beta=-2.0, relu=True, math=math,
               stage=3, expect_tc=None, seed=751))


def test_fp32_math_is_the_staged_cuda_core_call():
    M, N, K = 700, 500, 300
    g = torch.Generator().manual_seed(9)
    A = torch.rand(K, M, generator=g).cuda()
    B = torch.rand(K, N, generator=g).cuda()
    outs = []
    for call in ("math", "sgemm"):
        C = torch.full((M, N), float("nan"), device="cuda")
        need = fg.staged_workspace_size(1, 0, M, N, K, 1)
        ws = torch.empty(need // 4, device="cuda")
        args = (1, 0, M, N, K, 1.0, A, M, 0, B, N, 0, 0.0, C, N, 0, 1, None, False, -1, ws, need)
        if call == "math":
            assert fg.math_staged_workspace_size(fg.MATH_FP32, 1, 0, M, N, K, 1) == need
            fg.gemm_math_staged(fg.MATH_FP32, *args)
        else:
            fg.sgemm_staged(*args)
        torch.cuda.synchronize()
        outs.append(C)
    assert torch.equal(outs[0], outs[1])
