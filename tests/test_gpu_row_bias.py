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

# (M, N, K, offset of A) chosen so the selector lands on each configuration on a GPU
# with about 150 SMs (asserted below for the GPU at hand).
SHAPES = [
    (1600, 1600, 40, 0, "simt_128x128_t8x8_split"),
    (2000, 2100, 40, 0, "simt_128x128_t8x8"),
    (1024, 1000, 40, 0, "simt_128x64x16_t8x8_s4"),
    (832, 840, 36, 0, "simt_64x64x16_t4x4_s4"),
    (640, 640, 24, 0, "simt_32x32x16_t4x4_s4"),
    (100, 70, 33, 0, "simt_32x32x32_t4x4_s8_k4"),
    (130, 77, 45, 1, "simt_64x64x16_t4x4_s4_scalar"),
]


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("M,N,K,offA,name", SHAPES)
@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("relu", [False, True])
def test_row_bias_parity(M, N, K, offA, name, ta, tb, relu):
    if offA == 0:
        sms = _sms()
        if not 140 <= sms <= 160:
            pytest.skip("shape table assumes about 150 SMs")
        cfg = fg.select_config(ta, tb, M, N, K, 1, True, sms)
        if name.startswith("simt_128x128"):
            # whole tiles, or the last-wave split when tiles mod SMs is at most half the SMs
            r = (-(-M // 128) * -(-N // 128)) % sms
            name = "simt_128x128_t8x8" + ("_split" if 0 < r and 2 * r <= sms else "")
        assert fg.config_name(cfg) == name
    check(Case(ta=ta, tb=tb, M=M, N=N, K=K, alpha=1.0, beta=0.0, relu=relu, row_bias=True,
               offset=(offA, 0, 0), align_ld=offA == 0, seed=M + N + K))


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
