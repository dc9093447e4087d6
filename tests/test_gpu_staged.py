"""fgemm_sgemm_staged against the FP64 oracle.

The call copies operands into a caller workspace -- transposed k-major when stored with
k contiguous (A for op N, B for op T), row by row into aligned rows when already
k-major -- and runs the GEMM on the copies (GEMM 优化详解, "Level 1: Naive 实现":
re-store an operand that is read across its rows).  Checked here, through the C ABI:
every transpose layout with every copy mask and the model's own choice, ragged sizes
over several tiles, strided batches with and without a shared operand, unaligned
operands (the copies are aligned, so the vector kernels run), alpha = 0 and K = 0 (no
copies, no workspace read), beta = 0 over a NaN C, replay in a CUDA graph, a workspace
that bounds the model's choice, and the argument checks.  Integer data must come back
bit-exact, uniform data within 1e-5 * mag; the harness fills the workspace with NaN,
so any element the GEMM read before the copy wrote it would show.
"""

import itertools

import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
from gpu_harness import Case, check

pytestmark = pytest.mark.gpu

COMBOS = list(itertools.product((0, 1), (0, 1)))
STAGES = [fg.STAGE_AUTO, 0, 1, 2, 3]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    fg.library()


@pytest.mark.parametrize("stage", STAGES)
@pytest.mark.parametrize("ta,tb", COMBOS)
def test_every_layout_and_mask_integer_exact(ta, tb, stage):
    check(Case(ta=ta, tb=tb, M=300, N=260, K=333, alpha=1.5, beta=0.5, bias=True, relu=True,
               pad=(4, 8, 4), stage=stage, seed=100 + 10 * stage + 2 * ta + tb))


@pytest.mark.parametrize("ta,tb", COMBOS)
def test_whole_and_last_wave_tiles_uniform(ta, tb):
    # 1700 x 1650: 182 tiles of 128 x 128, so the GEMM after the copies runs whole tiles
    # and a last wave; uniform data against the 1e-5 * mag bound
    check(Case(ta=ta, tb=tb, M=1700, N=1650, K=300, alpha=-0.75, beta=1.25, ints=False,
               bias=True, stage=3, seed=120 + 2 * ta + tb))


@pytest.mark.parametrize("share", [(False, False), (True, False), (False, True)])
@pytest.mark.parametrize("ta,tb", [(0, 1), (0, 0), (1, 1)])
def test_strided_batch_and_shared_operands(ta, tb, share):
    # a shared operand (stride 0) is copied once and read by every problem
    check(Case(ta=ta, tb=tb, M=200, N=170, K=96, alpha=1.0, beta=-1.0, batch=6, stage=3,
               share_a=share[0], share_b=share[1], seed=130 + 2 * ta + tb + 7 * share[0]))


@pytest.mark.parametrize("stage", [fg.STAGE_AUTO, 3])
@pytest.mark.parametrize("ta,tb", COMBOS)
def test_unaligned_operands(ta, tb, stage):
    # odd leading dimensions and pointers 4 bytes past a 16-byte boundary: the plain call
    # would take the element-wise kernel; staged copies are aligned
    check(Case(ta=ta, tb=tb, M=333, N=222, K=111, alpha=2.0, beta=0.0, align_ld=False,
               pad=(1, 3, 1), offset=(1, 3, 2), stage=stage, seed=140 + 2 * ta + tb))


@pytest.mark.parametrize("ta,tb", COMBOS)
def test_no_products_reads_neither_operand_nor_workspace(ta, tb):
    # alpha = 0 (A holds NaN) and K = 0: the result is beta * C + bias, nothing copied
    check(Case(ta=ta, tb=tb, M=129, N=131, K=64, alpha=0.0, beta=0.5, a_nan=True, bias=True,
               stage=3, seed=150 + ta))
    check(Case(ta=ta, tb=tb, M=129, N=131, K=0, alpha=1.0, beta=-2.0, relu=True, stage=3,
               seed=155 + tb))


@pytest.mark.parametrize("ta,tb", COMBOS)
def test_beta_zero_never_reads_c(ta, tb):
    check(Case(ta=ta, tb=tb, M=260, N=300, K=200, alpha=1.0, beta=0.0, c_nan=True, stage=3,
               ints=False, seed=160 + 2 * ta + tb))


def test_staged_equals_plain_bit_for_bit_on_integers():
    # integer data: every partial sum is exact, so staged and plain agree in every bit
    M, N, K = 1024, 768, 512
    g = torch.Generator().manual_seed(7)
    A = torch.randint(-4, 5, (M, K), generator=g).float().cuda()
    B = torch.randint(-4, 5, (N, K), generator=g).float().cuda()
    plain = torch.empty(M, N, device="cuda")
    staged = torch.full((M, N), float("nan"), device="cuda")
    fg.gemm_explicit(-1, 0, 1, M, N, K, 1.0, A, K, 0, B, K, 0, 0.0, plain, N, 0, 1)
    need = fg.staged_workspace_size(0, 1, M, N, K, 1)
    ws = torch.empty(need // 4, device="cuda")
    fg.sgemm_staged(0, 1, M, N, K, 1.0, A, K, 0, B, K, 0, 0.0, staged, N, 0, 1, None, False, 3,
                    ws, need)
    torch.cuda.synchronize()
    assert torch.equal(plain, staged)


def test_staged_call_replays_in_a_cuda_graph():
    M, N, K = 500, 700, 300
    g = torch.Generator().manual_seed(8)
    A = torch.rand(M, K, generator=g).cuda()
    B = torch.rand(N, K, generator=g).cuda()
    need = fg.staged_workspace_size(0, 1, M, N, K, 1)
    ws = torch.empty(need // 4, device="cuda")
    eager, replayed = torch.empty(M, N, device="cuda"), torch.empty(M, N, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        fg.sgemm_staged(0, 1, M, N, K, 1.0, A, K, 0, B, K, 0, 0.0, eager, N, 0, 1, None, False, 3,
                        ws, need, stream=stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        fg.sgemm_staged(0, 1, M, N, K, 1.0, A, K, 0, B, K, 0, 0.0, replayed, N, 0, 1, None, False,
                        3, ws, need, stream=stream)
    replayed.fill_(float("nan"))
    ws.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(replayed, eager)


def test_argument_checks_launch_nothing():
    M, N, K = 256, 256, 256
    A = torch.ones(M, K, device="cuda")
    B = torch.ones(K, N, device="cuda")
    C = torch.full((M, N), 7.0, device="cuda")
    need_a = K * M * 4  # the copy of A alone
    ws = torch.empty(need_a // 4 + 4, device="cuda")
    bad = [
        dict(workspace=None, workspace_bytes=0, stage=1),  # forced copies need room
        dict(workspace=ws, workspace_bytes=need_a - 4, stage=1),
        dict(workspace=ws, workspace_bytes=need_a, stage=3),  # A fits, B does not
        dict(workspace=ws.data_ptr() + 4, workspace_bytes=need_a, stage=-1),  # misaligned
        dict(workspace=ws, workspace_bytes=need_a, stage=4),
        dict(workspace=ws, workspace_bytes=need_a, stage=-2),
    ]
    for kw in bad:
        st = fg.sgemm_staged(0, 0, M, N, K, 1.0, A, K, 0, B, N, 0, 0.0, C, N, 0, 1, None, False,
                             kw["stage"], kw["workspace"], kw["workspace_bytes"], check=False)
        assert st == fg.ERR_INVALID_VALUE, kw
    torch.cuda.synchronize()
    assert bool((C == 7.0).all())
    # the model's choice within whatever workspace there is: none at all, or one that
    # holds only the copy of A; stage = 0 runs the plain kernels without a workspace
    for stage, w, wb in ((-1, None, 0), (-1, ws, need_a), (1, ws, need_a), (0, None, 0)):
        C.fill_(7.0)
        fg.sgemm_staged(0, 0, M, N, K, 1.0, A, K, 0, B, N, 0, 0.0, C, N, 0, 1, None, False,
                        stage, w, wb)
        torch.cuda.synchronize()
        assert bool((C == float(K)).all()), (stage, wb)


@pytest.mark.parametrize("ta,tb", COMBOS)
def test_unaligned_operands_copied_by_the_model(ta, tb):
    # 1200^3 with odd leading dimensions: the model copies at least the k-major operands
    # (A for op T, B for op N: the plain kernels would move them element by element) into
    # aligned rows, and may transpose the others; NT has no k-major operand and needs none
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms == 152:
        mask = fg.staged_choice(ta, tb, 1200, 1200, 1200, 1, False, False, False, False, sms)
        k_major = (1 if ta == 1 else 0) | (2 if tb == 0 else 0)
        assert mask & k_major == k_major
    check(Case(ta=ta, tb=tb, M=1200, N=1200, K=1200, alpha=1.0, beta=0.5, bias=True,
               align_ld=False, pad=(1, 1, 0), stage=fg.STAGE_AUTO, seed=170 + 2 * ta + tb))


def test_model_choice_on_this_gpu():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms != 152:
        pytest.skip("expectations measured on 152 SMs")
    ch = lambda *a: fg.staged_choice(*a, False, False, True, True, sms)
    assert ch(0, 0, 4096, 4096, 4096, 1) == 1  # 4096^3: copy A
    assert ch(0, 0, 8192, 11008, 4096, 1) == 1  # the FC layer: copy X
    assert ch(0, 1, 2048, 2048, 128, 128) == 3  # batched Q K^T: copy both
    assert ch(0, 0, 2048, 128, 2048, 128) == 0  # Score x V: the 2 GiB of scores stay
    assert ch(0, 0, 1024, 1024, 1024, 1) == 0
    assert ch(0, 0, 256, 256, 256, 1) == 0
