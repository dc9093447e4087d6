"""fgemm_sgemm_splitk_noalloc: the split-K GEMM for callers that may not allocate
device memory (a plugin inside a program that owns all GPU memory through its own
pool, a latency-critical loop that cannot pay for cudaMalloc's synchronisation, a
process with a fixed memory budget).

The entry point keeps its partial products in the library's fixed device array
instead of a caller workspace.  Checked here, through the C ABI:
  * two calls in a row with different data and shapes (the array keeps the previous
    call's contents, which must not leak into the next result): each result matches
    the existing workspace entry point fgemm_sgemm_splitk within the parity tests'
    tolerance (in fact bit for bit: the same kernels in the same order), and every
    element matches the FP64 oracle within 1e-5 * mag;
  * the calls allocate no device memory (free memory is unchanged across them);
  * after a first call, a call captured in a CUDA graph replays to the same bits;
  * problems whose partial products do not fit are refused before anything runs,
    while calls that need no partial products run at any size.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test.
"""

import numpy as np
import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
import oracle
from dense_fp32_gemm_sm_gb300 import workloads

pytestmark = pytest.mark.gpu

REL_TOL = 1e-5
FLT_MIN = float(np.finfo(np.float32).tiny)

# (M, N, K, ta, tb, splits, relu): two different problems, back to back
CASES = [(1024, 1024, 1024, 0, 0, 4, False), (300, 500, 2000, 1, 1, 3, True)]


def _problem(seed, M, N, K, ta, tb):
    g = workloads.generator(seed)
    A = workloads.uniform(g, (K, M) if ta else (M, K))
    B = workloads.uniform(g, (N, K) if tb else (K, N))
    C0 = workloads.uniform(g, (M, N))
    bias = workloads.uniform(g, (N,))
    return A, B, C0, bias


def _within(got, want, mag):
    err = np.abs(got.astype(np.float64) - want)
    return bool((err <= REL_TOL * mag + FLT_MIN).all()), float((err / (mag + FLT_MIN)).max())


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    fg.library()


def test_noalloc_matches_workspace_entry_point_and_oracle_on_two_calls():
    prepared = []
    for i, (M, N, K, ta, tb, splits, relu) in enumerate(CASES):
        A, B, C0, bias = _problem(40 + i, M, N, K, ta, tb)
        assert 0 < fg.splitk_workspace_size(M, N, K, splits) <= fg.NOALLOC_SCRATCH_BYTES
        lda, ldb = A.shape[1], B.shape[1]
        d = dict(A=A.cuda(), B=B.cuda(), bias=bias.cuda(), ref=C0.cuda(), out=C0.cuda())
        need = fg.splitk_workspace_size(M, N, K, splits)
        d["ws"] = torch.empty(need // 4, device="cuda")
        prepared.append((M, N, K, ta, tb, splits, relu, lda, ldb, need, A, B, C0, bias, d))
    torch.cuda.synchronize()

    # the existing entry point, with a caller workspace
    for M, N, K, ta, tb, splits, relu, lda, ldb, need, A, B, C0, bias, d in prepared:
        fg.sgemm_splitk(ta, tb, M, N, K, 1.5, d["A"], lda, d["B"], ldb, 0.5, d["ref"], N,
                        d["bias"], relu, splits, d["ws"], need)
    torch.cuda.synchronize()
    # the entry point without allocation: two calls in a row through the same array
    for M, N, K, ta, tb, splits, relu, lda, ldb, need, A, B, C0, bias, d in prepared:
        fg.sgemm_splitk_noalloc(ta, tb, M, N, K, 1.5, d["A"], lda, d["B"], ldb, 0.5, d["out"], N,
                                d["bias"], relu, splits)
    torch.cuda.synchronize()
    for M, N, K, ta, tb, splits, relu, lda, ldb, need, A, B, C0, bias, d in prepared:
        got, ref = d["out"].cpu().numpy(), d["ref"].cpu().numpy()
        want, mag = oracle.gemm(ta, tb, M, N, K, 1.5, A.numpy().reshape(-1), lda,
                                B.numpy().reshape(-1), ldb, 0.5, C0.numpy().reshape(-1), N,
                                bias=bias.numpy(), relu=relu)
        ok, worst = _within(got, want, mag)
        assert ok, "no-alloc result outside 1e-5*mag of the oracle (worst %g)" % worst
        ok, worst = _within(ref, want, mag)
        assert ok, "workspace result outside 1e-5*mag of the oracle (worst %g)" % worst
        # against the existing entry point: within the parity tolerance, and the same bits
        assert (np.abs(got.astype(np.float64) - ref) <= REL_TOL * mag + FLT_MIN).all()
        assert np.array_equal(got, ref)


def test_noalloc_allocates_no_device_memory():
    M, N, K, ta, tb, splits, relu = CASES[0]
    A, B, C0, bias = _problem(50, M, N, K, ta, tb)
    dA, dB, dbias, dC = A.cuda(), B.cuda(), bias.cuda(), C0.cuda()

    def call():
        fg.sgemm_splitk_noalloc(ta, tb, M, N, K, 1.0, dA, K, dB, N, 0.0, dC, N, dbias, relu,
                                splits)

    call()  # first call in this context: the array's address is looked up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, "device memory changed by %d bytes" % (free0 - free1)


def test_noalloc_call_replays_in_a_cuda_graph():
    M, N, K, ta, tb, splits, relu = CASES[1]
    A, B, C0, bias = _problem(60, M, N, K, ta, tb)
    lda, ldb = A.shape[1], B.shape[1]
    dA, dB, dbias = A.cuda(), B.cuda(), bias.cuda()
    eager, replayed = torch.empty(M, N, device="cuda"), torch.empty(M, N, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        fg.sgemm_splitk_noalloc(ta, tb, M, N, K, 2.0, dA, lda, dB, ldb, 0.0, eager, N, dbias,
                                relu, splits, stream=stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        fg.sgemm_splitk_noalloc(ta, tb, M, N, K, 2.0, dA, lda, dB, ldb, 0.0, replayed, N, dbias,
                                relu, splits, stream=stream)
    replayed.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(replayed, eager)


def test_noalloc_rejects_problems_larger_than_the_array():
    M = N = 2048
    K, splits = 4096, 4  # 4 x 2048 x 2048 floats = 64 MiB of partial products
    assert fg.splitk_workspace_size(M, N, K, splits) > fg.NOALLOC_SCRATCH_BYTES
    A = torch.zeros(M * K, device="cuda")
    B = torch.zeros(K * N, device="cuda")
    C = torch.full((M, N), 7.0, device="cuda")
    st = fg.sgemm_splitk_noalloc(0, 0, M, N, K, 1.0, A, K, B, N, 0.0, C, N, None, False, splits,
                                 check=False)
    torch.cuda.synchronize()
    assert st == fg.ERR_NOT_SUPPORTED
    assert bool((C == 7.0).all())  # nothing ran


def test_noalloc_without_partial_products_runs_at_any_size():
    # splits == 1 and alpha == 0 use no partial products, so the array's size does not
    # limit them: the same result as the workspace entry point.
    M = N = 2048
    K = 4096
    g = workloads.generator(70)
    A, B = workloads.small_ints(g, (M, K)).cuda(), workloads.small_ints(g, (K, N)).cuda()
    C0 = workloads.small_ints(g, (M, N)).cuda()
    for alpha, splits in ((1.0, 1), (0.0, 4)):
        out, ref = C0.clone(), C0.clone()
        fg.sgemm_splitk_noalloc(0, 0, M, N, K, alpha, A, K, B, N, 0.5, out, N, None, False, splits)
        fg.sgemm_splitk(0, 0, M, N, K, alpha, A, K, B, N, 0.5, ref, N, None, False, splits, None, 0)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        if alpha == 0.0:
            assert torch.equal(out, 0.5 * C0)
