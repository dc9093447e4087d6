"""Row-broadcast bias epilogue (fgemm_sgemm_row_bias_relu) against the FP64 oracle.

The fused epilogue of GEMM 优化详解, "Level 6: Kernel Fusion" adds one bias value per
output column; this entry point adds one per output row, before the optional ReLU.
Sizes are picked so the shape-based selector lands on every tile configuration, and
integer-valued inputs make every comparison bit-exact.
"""

import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
from gpu_harness import Case, check

pytestmark = pytest.mark.gpu

# The row-bias entry point has no configuration argument: the selector picks one.
# For each configuration and layout the test takes the smallest shape of this list
# on which the selector, at this GPU's SM count, picks that configuration.
CANDIDATES = sorted(
    ((M, N, K) for K in (40, 64, 100, 256, 512, 2048) for M in range(96, 2500, 100)
     for N in (M, M + 36, 2 * M + 10)),
    key=lambda s: s[0] * s[1] * s[2])
TARGETS = ["simt_128x128_t8x8", "simt_128x128_t8x8_split", "simt_128x128_t8x8_ksplit",
           "simt_128x128_t8x8_kchain", "simt_128x64x16_t8x8_s4", "simt_64x64x16_t4x4_s4",
           "simt_32x32x16_t4x4_s4", "simt_32x32x32_t4x4_s8_k4"]
# The quarter-tile split wins only in narrow bands of the tile remainder (the k-chain
# takes most of them); where no candidate reaches it, its epilogue (the whole-tile one)
# is covered by the others.
OPTIONAL = {"simt_128x128_t8x8_split"}


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _shape_for(name, ta, tb):
    sms = _sms()
    for M, N, K in CANDIDATES:
        if fg.config_name(fg.select_config(ta, tb, M, N, K, 1, True, sms)) == name:
            return M, N, K
    if name in OPTIONAL:
        pytest.skip("the selector picks %s for no candidate in layout %d%d" % (name, ta, tb))
    raise AssertionError("the selector never picks %s for layout %d%d" % (name, ta, tb))


@pytest.mark.parametrize("name", TARGETS)
@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("relu", [False, True])
def test_row_bias_parity(name, ta, tb, relu):
    M, N, K = _shape_for(name, ta, tb)
    check(Case(ta=ta, tb=tb, M=M, N=N, K=K, alpha=1.0, beta=0.0, relu=relu, row_bias=True,
               seed=M + N + K))


@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_row_bias_unaligned_takes_the_scalar_config(ta, tb):
    assert fg.config_name(fg.select_config(ta, tb, 130, 77, 45, 1, False, _sms())).endswith(
        "_scalar")
    check(Case(ta=ta, tb=tb, M=130, N=77, K=45, relu=True, row_bias=True, offset=(1, 0, 0),
               align_ld=False, seed=252))


@pytest.mark.parametrize("alpha,beta", [(2.0, 1.0), (0.0, -1.0), (-1.0, 0.5)])
def test_row_bias_with_beta(alpha, beta):
    check(Case(M=257, N=129, K=67, alpha=alpha, beta=beta, relu=True, row_bias=True, seed=7))


def test_row_bias_k_zero():
    # No products: C = relu(beta*C + row_bias).
    check(Case(M=96, N=64, K=0, alpha=1.0, beta=1.0, relu=True, row_bias=True, seed=8))


def test_row_bias_real_values():
    check(Case(M=300, N=260, K=513, alpha=0.75, beta=0.25, relu=True, row_bias=True, ints=False,
               seed=9))


def test_row_bias_null_is_plain_gemm():
    # A NULL row bias leaves the plain fused-less GEMM.
    check(Case(M=200, N=120, K=50, relu=False, seed=10))
    M, N, K = 64, 48, 16
    A = torch.ones(M, K, device="cuda")
    B = torch.ones(K, N, device="cuda")
    C = torch.full((M, N), -5.0, device="cuda")
    fg.sgemm_row_bias_relu(0, 0, M, N, K, 1.0, A, K, B, N, 0.0, C, N, None, True)
    torch.cuda.synchronize()
    assert bool((C == float(K)).all())
