"""IEEE special values in the operands: NaN and +-Inf among small-integer entries.

Each output element is a sum of products (GEMM 优化详解, "数学定义"), so IEEE arithmetic
decides where NaN and infinities land: NaN times anything is NaN, an infinity times zero
is NaN, +Inf plus -Inf is NaN.  With every other entry a small integer no sum overflows
and none of this depends on the order of the sum, so the CUDA-core kernels must match the
FP64 oracle exactly, NaN for NaN and infinity for infinity: through every configuration,
the last-wave splits, the staged copies, split-K and ReLU (which maps NaN to 0, the
fmaxf reading).  TF32 reads Inf and the canonical quiet NaN unchanged, so it matches too.
3xTF32 splits each operand into a TF32 part and a residual and adds three products; the
correction products multiply one operand's residual by the other's high part, and an
integer's residual is 0, so an infinity becomes 0 x Inf = NaN there: every output the
definition makes non-finite must be non-finite, every finite one exact.

The special entries sit in the first and last rows and columns of the operands and in
the last k, so that they cross tile edges, the ragged tail and the k-split boundaries.
"""

import numpy as np
import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
import oracle
from dense_fp32_gemm_sm_gb300 import workloads
from gpu_harness import Case, run

pytestmark = pytest.mark.gpu

NAN, INF = float("nan"), float("inf")
M, N, K = 300, 260, 333
# (operand, row, column of op(A) = M x K or op(B) = K x N, value)
OP_SPECIALS = [("A", 5, 7, NAN), ("A", 299, 332, INF), ("A", 150, 200, -INF),
               ("B", 100, 259, -INF), ("B", 332, 0, INF), ("B", 17, 130, NAN)]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    fg.library()


def stored(ta, tb, specials=OP_SPECIALS):
    """The entries in stored coordinates: A is K x M for op T, B is N x K for op T."""
    out = []
    for which, r, c, v in specials:
        t = ta if which == "A" else tb
        out.append((which, c, r, v) if t else (which, r, c, v))
    return tuple(out)


def check_ieee(case, three=False):
    got, want, _, untouched_ok = run(case)
    assert untouched_ok, "the call wrote outside the M x N region of C"
    got = got.astype(np.float64)
    finite = np.isfinite(want)
    assert (~finite).any() and finite.any()
    if three:
        assert np.array_equal(got[finite], want[finite]), "a finite result differs"
        assert not np.isfinite(got[~finite]).any(), "a non-finite result came back finite"
        return
    bad = ~((got == want) | (np.isnan(got) & np.isnan(want)))
    assert not bad.any(), "%d of %d differ, first at %s: %r, the oracle says %r" % (
        bad.sum(), bad.size, tuple(np.argwhere(bad)[0]), got[bad][0], want[bad][0])


@pytest.mark.parametrize("config", range(10))
def test_every_configuration(config):
    assert fg.num_configs() == 10
    check_ieee(Case(ta=0, tb=0, M=M, N=N, K=K, alpha=1.5, beta=0.5, bias=True, config=config,
                    specials=stored(0, 0), seed=600 + config))


@pytest.mark.parametrize("relu", [False, True])
@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_layouts_and_relu(ta, tb, relu):
    check_ieee(Case(ta=ta, tb=tb, M=M, N=N, K=K, alpha=-1.0, beta=0.0, relu=relu, c_nan=True,
                    specials=stored(ta, tb), seed=610 + 2 * ta + tb))


def test_large_grid_with_last_wave():
    # 2000 x 1900: 240 tiles of 128 x 128, whole tiles and a last wave
    sp = [("A", 0, 0, NAN), ("A", 1999, 255, INF), ("B", 255, 1899, -INF), ("B", 100, 950, INF)]
    check_ieee(Case(ta=1, tb=0, M=2000, N=1900, K=256, alpha=1.0, beta=0.0,
                    specials=stored(1, 0, sp), seed=620))


@pytest.mark.parametrize("stage", [fg.STAGE_AUTO, 3])
def test_staged_batch(stage):
    check_ieee(Case(ta=0, tb=1, M=M, N=N, K=K, alpha=1.0, beta=-1.0, batch=2, stage=stage,
                    specials=stored(0, 1), seed=630))


@pytest.mark.parametrize("math", [fg.MATH_TF32, fg.MATH_3XTF32], ids=["tf32", "3xtf32"])
@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1)])
def test_tensor_cores(math, ta, tb):
    check_ieee(Case(ta=ta, tb=tb, M=M, N=N, K=K, alpha=2.0, beta=0.5, math=math,
                    specials=stored(ta, tb), seed=640 + 2 * ta + tb),
               three=math == fg.MATH_3XTF32)


def test_split_k():
    g = workloads.generator(650)
    A = workloads.small_ints(g, (M, K)).numpy()
    B = workloads.small_ints(g, (K, N)).numpy()
    C0 = workloads.small_ints(g, (M, N)).numpy()
    bias = workloads.small_ints(g, (N,)).numpy()
    for which, r, c, v in OP_SPECIALS:
        (A if which == "A" else B)[r, c] = v
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C0))
    dbias = torch.from_numpy(bias).cuda()
    need = fg.splitk_workspace_size(M, N, K, 4)
    ws = torch.full((need // 4,), NAN, device="cuda")
    fg.sgemm_splitk(0, 0, M, N, K, 1.0, dA, K, dB, N, 0.5, dC, N, dbias, False, 4, ws, need)
    torch.cuda.synchronize()
    got = dC.cpu().numpy().astype(np.float64)
    want, _ = oracle.gemm(0, 0, M, N, K, 1.0, A.reshape(-1), K, B.reshape(-1), N, beta=0.5,
                          C0=C0.reshape(-1), ldc=N, bias=bias, want_mag=False)
    assert (~np.isfinite(want)).any()
    assert np.array_equal(got, want, equal_nan=True)
