"""CUDA library vs the FP64 oracle, element by element, on seeded inputs.

Every kernel configuration runs every transpose combination on shapes that
span several CTA tiles with ragged M, N and K tails, with small-integer data
(bit-exact) and uniform data (1e-5 * mag).  Edge cases: 1x1x1, K = 0,
alpha = 0 (A not read), beta = 0 (C not read), all four bias/ReLU
combinations, padded leading dimensions, unaligned pointers, strided batches.
"""

import itertools

import numpy as np
import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
from gpu_harness import Case, check

pytestmark = pytest.mark.gpu

COMBOS = list(itertools.product((0, 1), (0, 1)))
VEC_CONFIGS = [0, 1, 2, 4, 5, 6, 7, 8]
SCALAR_CONFIG = 3       # 64 x 64, element-wise copies
SCALAR_CONFIGS = [3, 9]  # and the 128 x 128 tile with element-wise copies
SHAPES = [(300, 200, 130), (1, 1, 1), (129, 65, 17), (64, 128, 3), (7, 333, 64), (257, 31, 515)]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    fg.library()


def test_config_names_match_ids():
    assert all(fg.config_name(c).endswith("_scalar") for c in SCALAR_CONFIGS)
    assert all(not fg.config_name(c).endswith("_scalar") for c in VEC_CONFIGS)
    assert sorted(VEC_CONFIGS + SCALAR_CONFIGS) == list(range(fg.num_configs()))


@pytest.mark.parametrize("config", VEC_CONFIGS + SCALAR_CONFIGS)
@pytest.mark.parametrize("ta,tb", COMBOS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_integer_exact(config, ta, tb, shape):
    M, N, K = shape
    check(Case(ta=ta, tb=tb, M=M, N=N, K=K, alpha=2.0, beta=-0.5, config=config,
               pad=(4, 8, 4), seed=M + N + K))


@pytest.mark.parametrize("config", VEC_CONFIGS + SCALAR_CONFIGS)
@pytest.mark.parametrize("ta,tb", COMBOS)
def test_uniform_floats(config, ta, tb):
    check(Case(ta=ta, tb=tb, M=515, N=387, K=1029, alpha=1.5, beta=0.5, ints=False,
               config=config, seed=3))


@pytest.mark.parametrize("config", VEC_CONFIGS + SCALAR_CONFIGS)
@pytest.mark.parametrize("bias,relu", [(False, False), (True, False), (False, True), (True, True)])
def test_bias_relu_combinations(config, bias, relu):
    for ta, tb in COMBOS:
        check(Case(ta=ta, tb=tb, M=200, N=152, K=40, bias=bias, relu=relu, config=config, seed=7))


@pytest.mark.parametrize("ta,tb", COMBOS)
def test_unaligned_pointers_and_ld_use_scalar_path(ta, tb):
    for offset, pad in (((1, 0, 0), (0, 0, 0)), ((0, 3, 0), (1, 0, 0)), ((2, 1, 3), (1, 3, 1))):
        check(Case(ta=ta, tb=tb, M=150, N=90, K=77, alpha=1.0, beta=1.0, offset=offset, pad=pad,
                   config=-1, seed=11, align_ld=False))
        for config in SCALAR_CONFIGS:
            check(Case(ta=ta, tb=tb, M=150, N=90, K=77, ints=False, offset=offset, pad=pad,
                       config=config, seed=12, align_ld=False))


@pytest.mark.parametrize("ta,tb", COMBOS)
def test_unaligned_large_problem_takes_the_128_tile(ta, tb):
    # Odd leading dimensions at 2600 x 2400 x 900: the selector picks the 128 x 128 tile
    # with element-wise copies (whole and ragged tiles), bit-exact on integers
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms == 152:
        assert fg.select_config(ta, tb, 2600, 2400, 900, 1, False, sms) == 9
    check(Case(ta=ta, tb=tb, M=2600, N=2400, K=900, alpha=2.0, beta=-1.0, bias=True, relu=True,
               offset=(1, 2, 3), pad=(1, 1, 1), config=-1, seed=13 + 2 * ta + tb,
               align_ld=False))


@pytest.mark.parametrize("config", [-1, 0, 1, 7, 8])
@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1), (1, 1)])
def test_unaligned_k_contiguous_operand_keeps_the_vector_kernels(config, ta, tb):
    # Operands stored with k contiguous (A for op N, B for op T) are copied element by
    # element in every configuration, so their alignment does not matter: odd leading
    # dimensions and shifted pointers on them run the 16-byte-vector configurations.
    off_a, pad_a = (1, 1) if ta == 0 else (0, 0)
    off_b, pad_b = (2, 3) if tb == 1 else (0, 0)
    if config < 0 and torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert not fg.config_name(fg.select_config(ta, tb, 1500, 1400, 300, 1, True,
                                                   152)).endswith("_scalar")
    check(Case(ta=ta, tb=tb, M=1500, N=1400, K=300, alpha=1.5, beta=0.5, bias=True,
               offset=(off_a, off_b, 0), pad=(pad_a, pad_b, 0), align_ld=False, config=config,
               seed=21 + 2 * ta + tb))


@pytest.mark.parametrize("config", [-1] + VEC_CONFIGS)
def test_unaligned_c_only(config):
    # A and B aligned, C shifted by one element: vector configs fall back to scalar stores.
    check(Case(M=130, N=72, K=48, beta=2.0, offset=(0, 0, 1), pad=(0, 0, 1), config=config,
               align_ld=False))


@pytest.mark.parametrize("config", VEC_CONFIGS + SCALAR_CONFIGS)
def test_k_zero_and_alpha_zero(config):
    check(Case(M=70, N=90, K=0, alpha=3.0, beta=-2.0, bias=True, relu=True, config=config))
    check(Case(M=70, N=90, K=33, alpha=0.0, beta=0.5, a_nan=True, config=config))


@pytest.mark.parametrize("config", VEC_CONFIGS + SCALAR_CONFIGS)
def test_beta_zero_never_reads_c(config):
    check(Case(M=96, N=80, K=24, beta=0.0, c_nan=True, bias=True, config=config))


@pytest.mark.parametrize("config", VEC_CONFIGS + SCALAR_CONFIGS)
@pytest.mark.parametrize("ta,tb", COMBOS)
def test_strided_batched(config, ta, tb):
    check(Case(ta=ta, tb=tb, M=70, N=130, K=45, alpha=0.5, beta=1.0, batch=3, config=config,
               seed=5))


def test_batched_broadcast_and_interleaved_c():
    # B shared by every problem (strideB = 0), C interleaved: row r of problem b
    # at C[r * (batch*N) + b*N].  Compared against one plain call per problem.
    batch, M, N, K = 4, 33, 20, 19
    g = torch.Generator().manual_seed(9)
    A = torch.randint(-4, 5, (batch, M, K), generator=g).float().cuda()
    B = torch.randint(-4, 5, (K, N), generator=g).float().cuda()
    C = torch.full((M, batch * N), float("nan"), device="cuda")
    fg.sgemm_strided_batched(0, 0, M, N, K, 1.0, A, K, M * K, B, N, 0, 0.0, C, batch * N, N, batch)
    for b in range(batch):
        ref = torch.full((M, N), float("nan"), device="cuda")
        fg.sgemm(0, 0, M, N, K, 1.0, A[b], K, B, N, 0.0, ref, N)
        torch.cuda.synchronize()
        assert torch.equal(C[:, b * N:(b + 1) * N], ref)
        want = (A[b].double().cpu() @ B.double().cpu()).float()
        assert torch.equal(ref.cpu(), want)


def test_entry_points_agree_with_explicit():
    # The three plain entry points reach the same kernels as gemm_explicit.
    M, N, K = 190, 210, 70
    g = torch.Generator().manual_seed(1)
    A = torch.randint(-4, 5, (M, K), generator=g).float().cuda()
    B = torch.randint(-4, 5, (K, N), generator=g).float().cuda()
    bias = torch.randint(-4, 5, (N,), generator=g).float().cuda()
    C1 = torch.zeros(M, N, device="cuda")
    C2 = torch.zeros(M, N, device="cuda")
    C3 = torch.zeros(M, N, device="cuda")
    fg.sgemm_bias_relu(0, 0, M, N, K, 1.0, A, K, B, N, 0.0, C1, N, bias, True)
    fg.gemm_explicit(-1, 0, 0, M, N, K, 1.0, A, K, 0, B, N, 0, 0.0, C2, N, 0, 1, bias, True)
    fg.sgemm(0, 0, M, N, K, 1.0, A, K, B, N, 0.0, C3, N)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
    assert torch.equal(C1, torch.clamp(C3 + bias, min=0.0))


def test_rejects_vector_config_on_unaligned_device_pointer():
    # A vector configuration refuses an unaligned k-major operand (B for op N, which it
    # moves in 16-byte copies) and accepts an unaligned k-contiguous one (A for op N,
    # copied element by element).
    X = torch.zeros(65, device="cuda")
    C = torch.full((4, 4), 7.0, device="cuda")
    st = fg.gemm_explicit(0, 0, 0, 4, 4, 4, 1.0, X, 4, 0, X.data_ptr() + 4, 4, 0, 0.0, C, 4, 0, 1,
                          check=False)
    assert st == fg.ERR_NOT_SUPPORTED
    st = fg.gemm_explicit(0, 0, 0, 4, 4, 4, 1.0, X.data_ptr() + 4, 4, 0, X, 4, 0, 0.0, C, 4, 0, 1,
                          check=False)
    torch.cuda.synchronize()
    assert st == fg.OK and bool((C == 0.0).all())

