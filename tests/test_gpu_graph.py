"""Library calls captured in a CUDA graph and replayed, against the same calls run eagerly.

Every call is asynchronous on the caller's stream and allocates nothing, so it can be
captured.  The cases cover one launch per call (whole tiles), the two-launch last-wave
splits (quarter tiles, and k-slice clusters launched with a cluster dimension), the
split-K path with its reduction kernel, the tensor-core kernel, and the staged
tensor-core call (a copy kernel, then the tensor-core kernel); replays must give
the eager result bit for bit, and integer data makes both exact.
"""

import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    fg.library()


def _config(name):
    return [i for i in range(fg.num_configs()) if fg.config_name(i) == name][0]


def _ints(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(-4, 5, shape, generator=g).float().cuda()


def _capture_and_compare(call, out):
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        call()  # one-time setup (kernel attributes) happens outside the capture
    torch.cuda.synchronize()
    eager = out.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    out.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        graph.replay()
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


@pytest.mark.parametrize("name", ["simt_128x128_t8x8", "simt_128x128_t8x8_split",
                                  "simt_128x128_t8x8_ksplit", "simt_128x128_t8x8_kchain",
                                  "simt_32x32x32_t4x4_s8_k4"])
def test_explicit_configs_replay(name):
    M, N, K = 1700, 1652, 200  # 182 tiles of 128 x 128: whole tiles and a last wave
    A, B, bias = _ints((M, K), 1), _ints((K, N), 2), _ints((N,), 3)
    C = torch.empty(M, N, device="cuda")
    cfg = _config(name)
    _capture_and_compare(
        lambda: fg.gemm_explicit(cfg, 0, 0, M, N, K, 1.0, A, K, 0, B, N, 0, 0.0, C, N, 0, 1, bias,
                                 True), C)
    want = torch.clamp((A.double() @ B.double()) + bias.double(), min=0).float()
    assert torch.equal(C, want)


def test_selected_call_replays_and_matches():
    # a batch of 5 problems: the selector's choice, whatever it is, captured
    b, M, N, K = 5, 1000, 992, 96
    A, B = _ints((b, M, K), 4), _ints((b, K, N), 5)
    C = torch.empty(b, M, N, device="cuda")
    _capture_and_compare(
        lambda: fg.sgemm_strided_batched(0, 0, M, N, K, 2.0, A, K, M * K, B, N, K * N, 0.0, C, N,
                                         M * N, b), C)
    assert torch.equal(C, (2.0 * torch.bmm(A.double(), B.double())).float())


def test_splitk_replays():
    M, N, K = 512, 384, 1000
    A, B = _ints((M, K), 6), _ints((K, N), 7)
    C = torch.empty(M, N, device="cuda")
    ws = torch.empty(fg.splitk_workspace_size(M, N, K, 4) // 4, device="cuda")
    _capture_and_compare(
        lambda: fg.sgemm_splitk(0, 0, M, N, K, 1.0, A, K, B, N, 0.0, C, N, None, False, 4, ws,
                                ws.numel() * 4), C)
    assert torch.equal(C, (A.double() @ B.double()).float())


@pytest.mark.parametrize("math", ["tf32", "3xtf32"])
def test_tensor_core_path_replays(math):
    M, N, K = 640, 768, 256
    A, B = _ints((M, K), 8), _ints((K, N), 9)
    C = torch.empty(M, N, device="cuda")
    mode = fg.MATH_TF32 if math == "tf32" else fg.MATH_3XTF32
    assert fg.math_supported(mode, 0, 0, M, N, K, 1.0, A, K, 0, B, N, 0, 1) == 1
    _capture_and_compare(
        lambda: fg.gemm_math(mode, 0, 0, M, N, K, 1.0, A, K, 0, B, N, 0, 0.0, C, N, 0, 1), C)
    # small integers are exact in TF32
    assert torch.equal(C, (A.double() @ B.double()).float())


@pytest.mark.parametrize("math", ["tf32", "3xtf32"])
def test_staged_tensor_core_call_replays(math):
    # TN: the copy of A (K x M stored) into the workspace, then the tensor-core kernel
    M, N, K = 640, 768, 256
    At, B = _ints((K, M), 10), _ints((K, N), 11)
    C = torch.empty(M, N, device="cuda")
    mode = fg.MATH_TF32 if math == "tf32" else fg.MATH_3XTF32
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert fg.math_staged_choice(mode, 1, 0, M, N, K, 1, False, False, True, True, sms) == 1
    need = fg.math_staged_workspace_size(mode, 1, 0, M, N, K, 1)
    ws = torch.empty(need // 4, device="cuda")
    _capture_and_compare(
        lambda: fg.gemm_math_staged(mode, 1, 0, M, N, K, 1.0, At, M, 0, B, N, 0, 0.0, C, N, 0, 1,
                                    None, False, fg.STAGE_AUTO, ws, need), C)
    assert torch.equal(C, (At.double().t() @ B.double()).float())
