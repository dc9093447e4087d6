"""The C-ABI library without a GPU: it loads, exports every declared symbol,
validates arguments before touching CUDA, and selects configurations."""

import os
import re

import pytest

import dense_fp32_gemm_sm_gb300 as fg

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "fgemm.h")
FAKE = 0x10000  # a non-null address that validation never dereferences


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fgemm_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol():
    lib = fg.library()
    names = declared_functions()
    assert "fgemm_sgemm" in names and "fgemm_sgemm_strided_batched" in names
    for name in names:
        assert hasattr(lib, name), name


def test_status_strings():
    for s in (fg.OK, fg.ERR_INVALID_VALUE, fg.ERR_LAUNCH, fg.ERR_NOT_SUPPORTED):
        assert fg.status_string(s).startswith("FGEMM_")
    assert "unknown" in fg.status_string(99)


def test_config_table():
    n = fg.num_configs()
    assert n >= 4
    names = [fg.config_name(i) for i in range(n)]
    assert all(names) and len(set(names)) == n
    assert fg.config_name(-1) is None and fg.config_name(n) is None


def _sgemm(**kw):
    args = dict(transa=0, transb=0, M=4, N=4, K=4, alpha=1.0, A=FAKE, lda=4, B=FAKE, ldb=4,
                beta=0.0, C=FAKE, ldc=4)
    args.update(kw)
    return fg.sgemm(**args, check=False)


@pytest.mark.parametrize("kw", [
    dict(transa=2), dict(transb=-1), dict(M=-1), dict(N=-1), dict(K=-1),
    dict(lda=3), dict(ldb=3), dict(ldc=3),
    dict(transa=1, M=8, lda=7), dict(transb=1, K=9, lda=9, ldb=8),
    dict(A=None), dict(B=None), dict(C=None),
])
def test_invalid_arguments_rejected_before_launch(kw):
    assert _sgemm(**kw) == fg.ERR_INVALID_VALUE


@pytest.mark.parametrize("kw", [dict(M=0), dict(N=0), dict(M=0, A=None, B=None, C=None)])
def test_empty_problems_are_noops(kw):
    assert _sgemm(**kw) == fg.OK


def test_ld_minimum_is_one_for_empty_rows():
    # K == 0 with lda == 0 is still invalid: ld >= max(1, stored row length).
    assert _sgemm(K=0, lda=0) == fg.ERR_INVALID_VALUE


def _batched(**kw):
    args = dict(transa=0, transb=0, M=4, N=4, K=4, alpha=1.0, A=FAKE, lda=4, strideA=16, B=FAKE,
                ldb=4, strideB=16, beta=0.0, C=FAKE, ldc=4, strideC=16, batch=3)
    args.update(kw)
    return fg.sgemm_strided_batched(**args, check=False)


@pytest.mark.parametrize("kw", [
    dict(batch=-1), dict(strideA=-4), dict(strideB=-4), dict(strideC=-4),
    dict(strideC=0), dict(strideC=15), dict(strideC=4, ldc=4),  # overlapping C problems
    dict(ldc=8, strideC=5),  # problem 1 starts inside row 0 of problem 0
])
def test_batched_rejects(kw):
    assert _batched(**kw) == fg.ERR_INVALID_VALUE


def test_batched_empty_is_noop():
    assert _batched(batch=0) == fg.OK
    assert _batched(batch=0, strideC=0) == fg.OK


def test_explicit_rejects_bad_config():
    st = fg.gemm_explicit(fg.num_configs(), 0, 0, 4, 4, 4, 1.0, FAKE, 4, 0, FAKE, 4, 0, 0.0, FAKE,
                          4, 0, 1, check=False)
    assert st == fg.ERR_INVALID_VALUE


def test_explicit_vector_config_refuses_unaligned():
    # A 16-byte-vector configuration with an unaligned k-major operand (the one it moves in
    # 16-byte copies: B for op N, A for op T): refused before launch.  (An unaligned
    # operand stored with k contiguous is copied element by element and accepted; the GPU
    # tests run that.)
    st = fg.gemm_explicit(0, 0, 0, 4, 4, 4, 1.0, FAKE, 4, 0, FAKE + 4, 4, 0, 0.0, FAKE, 4, 0, 1,
                          check=False)
    assert st == fg.ERR_NOT_SUPPORTED
    st = fg.gemm_explicit(0, 0, 0, 4, 4, 4, 1.0, FAKE, 4, 0, FAKE, 5, 0, 0.0, FAKE, 4, 0, 1,
                          check=False)
    assert st == fg.ERR_NOT_SUPPORTED
    st = fg.gemm_explicit(0, 1, 0, 4, 4, 4, 1.0, FAKE + 4, 4, 0, FAKE, 4, 0, 0.0, FAKE, 4, 0, 1,
                          check=False)
    assert st == fg.ERR_NOT_SUPPORTED
    st = fg.gemm_explicit(0, 1, 1, 4, 4, 4, 1.0, FAKE, 5, 0, FAKE + 4, 5, 0, 0.0, FAKE, 4, 0, 1,
                          check=False)
    assert st == fg.ERR_NOT_SUPPORTED


def test_selector():
    sel = fg.select_config
    name = lambda *a: fg.config_name(sel(*a))
    scalar = [i for i in range(fg.num_configs()) if fg.config_name(i).endswith("_scalar")]
    assert sel(0, 0, 4096, 4096, 4096, 1, 0, 152) in scalar
    # Choices of the fitted launch-time model on 152 SMs (each measured fastest, or
    # within 1 %, on a GB300):
    assert name(0, 0, 4096, 4096, 4096, 1, 1, 152) == "simt_128x128_t8x8_kchain"  # r = 112
    assert name(0, 1, 4096, 4096, 4096, 1, 1, 152) == "simt_128x128_t8x8_kchain"
    assert name(0, 0, 4096, 4864, 4096, 1, 1, 152) == "simt_128x128_t8x8"  # 8 x 152 tiles
    assert name(0, 0, 4096, 3648, 4096, 1, 1, 152) == "simt_128x128_t8x8_ksplit"  # r = 16
    assert name(0, 0, 8192, 11008, 4096, 1, 1, 152) == "simt_128x128_t8x8_ksplit"  # r = 32
    # the k-chain in as many slices as the model finds fastest (3072^3 measured 898 us
    # in five slices against 929 us as cluster k-split; 1792^2 x 1024 128 against 144 us
    # in three; 1280^2 x 4096, no whole tiles, 233 against 249 us in three)
    assert name(0, 0, 3072, 3072, 3072, 1, 1, 152) == "simt_128x128_t8x8_kchain"  # r = 120
    assert name(0, 0, 2048, 2048, 2048, 1, 1, 152) == "simt_128x128_t8x8_ksplit"  # r = 104
    assert name(0, 0, 1792, 1792, 1024, 1, 1, 152) == "simt_128x128_t8x8_kchain"  # r = 44
    assert name(0, 0, 1280, 1280, 4096, 1, 1, 152) == "simt_128x128_t8x8_kchain"  # 100 tiles
    assert name(0, 0, 1700, 1652, 4096, 1, 1, 152) == "simt_128x128_t8x8_ksplit"  # r = 30
    assert name(0, 0, 768, 768, 768, 1, 1, 152) == "simt_128x128_t8x8_ksplit"  # 36 tiles
    assert name(0, 0, 768, 768, 128, 1, 1, 152) == "simt_64x64x16_t4x4_s4"
    assert name(0, 0, 640, 640, 256, 1, 1, 152) == "simt_32x32x16_t4x4_s4"
    assert name(0, 0, 256, 256, 256, 1, 1, 152) == "simt_32x32x32_t4x4_s8_k4"
    # batches: QK^T (32768 tiles, r = 88, K = 128) whole; Score x V (2048 tiles, r = 72)
    assert name(0, 1, 2048, 2048, 128, 128, 1, 152) == "simt_128x128_t8x8"
    assert name(0, 0, 2048, 128, 2048, 128, 1, 152) == "simt_128x128_t8x8_ksplit"
    # the SM count enters: 1024 tiles on 148 SMs leave r = 136, which the k-chain would
    # run in four CTAs per SM; the cluster k-split is estimated faster there
    assert name(0, 0, 4096, 4096, 4096, 1, 1, 148) == "simt_128x128_t8x8_ksplit"
    assert sel(0, 0, -1, 4, 4, 1, 1, 152) == -1
    for ta in (0, 1):
        for tb in (0, 1):
            for n in (1, 7, 64, 255, 1000, 5000):
                for k in (0, 1, 100, 5000):
                    for sms in (1, 16, 152, 1000):
                        c = sel(ta, tb, n, n, k, 1, 1, sms)
                        assert 0 <= c < fg.num_configs() and c not in scalar


def test_gemm_math_validates_before_launch():
    st = fg.gemm_math(fg.MATH_3XTF32, 0, 1, -1, 4, 4, 1.0, FAKE, 4, 0, FAKE, 4, 0, 0.0, FAKE, 4, 0,
                      1, check=False)
    assert st == fg.ERR_INVALID_VALUE
    st = fg.gemm_math(9, 0, 1, 4, 4, 4, 1.0, FAKE, 4, 0, FAKE, 4, 0, 0.0, FAKE, 4, 0, 1,
                      check=False)
    assert st == fg.ERR_INVALID_VALUE
    st = fg.gemm_math(fg.MATH_TF32, 0, 1, 0, 4, 4, 1.0, FAKE, 4, 0, FAKE, 4, 0, 0.0, FAKE, 4, 0, 1,
                      check=False)
    assert st == fg.OK


def test_splitk_workspace_size():
    assert fg.splitk_workspace_size(4, 8, 100, 1) == 4 * 8 * 4
    # K = 100 in 4 slices -> slices of 32: ceil(100/32) = 4 slices
    assert fg.splitk_workspace_size(4, 8, 100, 4) == 4 * 4 * 8 * 4
    # K = 64 in 4 slices -> slices of 32: only 2 slices are used
    assert fg.splitk_workspace_size(4, 8, 64, 4) == 2 * 4 * 8 * 4
    assert fg.splitk_workspace_size(4, 8, 0, 4) == 0
    assert fg.splitk_workspace_size(-1, 8, 64, 4) == 0
    assert fg.splitk_workspace_size(4, 8, 64, 0) == 0
    assert fg.splitk_workspace_size(4, 8, 64, 65) == 0
    # sizes no allocation could hold saturate instead of wrapping around
    assert fg.splitk_workspace_size(2**31 - 1, 2**31 - 1, 2**31 - 1, 64) == 2**64 - 1


def test_splitk_rejects_missing_workspace_before_launch():
    args = (0, 0, 64, 64, 256, 1.0, FAKE, 256, FAKE, 64, 0.0, FAKE, 64, None, 0)
    assert fg.sgemm_splitk(*args, 4, None, 0, check=False) == fg.ERR_INVALID_VALUE
    need = fg.splitk_workspace_size(64, 64, 256, 4)
    assert fg.sgemm_splitk(*args, 4, FAKE, need - 4, check=False) == fg.ERR_INVALID_VALUE
    assert fg.sgemm_splitk(*args, 0, FAKE, need, check=False) == fg.ERR_INVALID_VALUE
    assert fg.sgemm_splitk(*args, 65, FAKE, need, check=False) == fg.ERR_INVALID_VALUE
    bad_ld = (0, 0, 64, 64, 256, 1.0, FAKE, 255, FAKE, 64, 0.0, FAKE, 64, None, 0)
    assert fg.sgemm_splitk(*bad_ld, 4, FAKE, need, check=False) == fg.ERR_INVALID_VALUE


@pytest.mark.parametrize("kw", [dict(M=-1), dict(ldc=3), dict(transa=1, M=8, lda=7), dict(C=None)])
def test_row_bias_entry_validates_before_launch(kw):
    args = dict(transa=0, transb=0, M=4, N=4, K=4, alpha=1.0, A=FAKE, lda=4, B=FAKE, ldb=4,
                beta=0.0, C=FAKE, ldc=4, row_bias=FAKE, apply_relu=True)
    assert fg.sgemm_row_bias_relu(**dict(args, M=0), check=False) == fg.OK
    args.update(kw)
    assert fg.sgemm_row_bias_relu(**args, check=False) == fg.ERR_INVALID_VALUE


def test_selector_extreme_arguments():
    # Sizes no allocation could hold still get a valid configuration (host-only call),
    # and a grid that divides evenly over the SMs never takes a last-wave split.
    sel = fg.select_config
    big = 2**31 - 1
    for args in ((big, big, big, big), (big, 1, 1, big), (1, 1, big, 1), (big, big, 0, 1)):
        for sms in (1, 152, 1000):
            c = sel(0, 0, *args, 1, sms)
            assert 0 <= c < fg.num_configs()
    for M, N, b in ((128 * 152, 128, 1), (128 * 19, 128 * 8, 1), (128, 128, 152 * 3)):
        assert (-(-M // 128) * -(-N // 128) * b) % 152 == 0
        assert not fg.config_name(sel(0, 0, M, N, 4096, b, 1, 152)).endswith("split")


def test_math_supported_host_query():
    q = fg.math_supported
    # FP32 is always what it says; an unknown arithmetic is -1
    assert q(fg.MATH_FP32, 0, 0, 4, 4, 4, 1.0, FAKE + 4, 5, 0, FAKE, 4, 0, 1) == 1
    assert q(7, 0, 0, 4, 4, 4, 1.0, FAKE, 4, 0, FAKE, 4, 0, 1) == -1
    for math in (fg.MATH_TF32, fg.MATH_3XTF32):
        # calls the tensor-core kernel cannot take fall back to the CUDA cores
        assert q(math, 0, 0, 4, 4, 4, 1.0, FAKE + 4, 4, 0, FAKE, 4, 0, 1) == 0  # A unaligned
        assert q(math, 0, 0, 4, 4, 4, 1.0, FAKE, 4, 0, FAKE, 5, 0, 1) == 0  # ldb not x4
        assert q(math, 0, 0, 4, 4, 4, 1.0, FAKE, 4, 6, FAKE, 4, 16, 2) == 0  # strideA not x4
        assert q(math, 0, 0, 4, 4, 0, 1.0, FAKE, 4, 0, FAKE, 4, 0, 1) == 0  # K == 0
        assert q(math, 0, 0, 4, 4, 4, 0.0, FAKE, 4, 0, FAKE, 4, 0, 1) == 0  # alpha == 0
        assert q(math, 0, 0, 0, 4, 4, 1.0, FAKE, 4, 0, FAKE, 4, 0, 1) == 0  # empty


def test_noalloc_checks_arguments_before_the_scratch_size():
    # 4 slices of a 2048 x 2048 C need 64 MiB of partial products, more than the array
    # holds: a valid call is refused as not supported, an invalid one as invalid --
    # both before any CUDA call.
    M = N = 2048
    K, splits = 4096, 4
    assert fg.splitk_workspace_size(M, N, K, splits) > fg.NOALLOC_SCRATCH_BYTES
    ok = dict(transa=0, transb=0, M=M, N=N, K=K, alpha=1.0, A=FAKE, lda=K, B=FAKE, ldb=N,
              beta=0.0, C=FAKE, ldc=N, bias=None, apply_relu=False, splits=splits)
    assert fg.sgemm_splitk_noalloc(**ok, check=False) == fg.ERR_NOT_SUPPORTED
    for bad in (dict(ldc=N - 1), dict(lda=K - 1), dict(M=-1), dict(splits=0), dict(splits=65),
                dict(C=None), dict(A=None)):
        assert fg.sgemm_splitk_noalloc(**dict(ok, **bad), check=False) == fg.ERR_INVALID_VALUE
    # nothing to do is a no-op at any size
    assert fg.sgemm_splitk_noalloc(**dict(ok, M=0), check=False) == fg.OK


def test_staged_workspace_size():
    sz = fg.staged_workspace_size
    # room for a copy of each operand: K rows of ld4(M) (A) and of ld4(N) (B) floats a
    # problem, B's at the next multiple of 256 bytes
    assert sz(0, 0, 4096, 4096, 4096, 1) == 2 * 4096 * 4096 * 4
    a = 2 * 3 * 8 * 4  # ld4(5) = 8, two problems, K = 3
    b = 2 * 3 * 8 * 4  # ld4(7) = 8
    for ta in (0, 1):
        for tb in (0, 1):
            assert sz(ta, tb, 5, 7, 3, 2) == (a + 255) // 256 * 256 + b
    for bad in ((0, 0, -1, 4, 4, 1), (0, 0, 4, 4, 0, 1), (0, 0, 4, 4, 4, 0), (2, 0, 4, 4, 4, 1)):
        assert sz(*bad) == 0
    # sizes no allocation could hold saturate instead of wrapping around
    big = 2**31 - 1
    assert sz(0, 0, big, big, big, big) == 2**64 - 1


def test_staged_choice_host_query():
    ch = fg.staged_choice  # the last argument, when given, is the workspace size
    # the model on 152 SMs: copy where the 16-byte-copy layout repays the copy
    assert ch(0, 0, 4096, 4096, 4096, 1, 0, 0, 1, 1, 152) == 1
    assert ch(0, 1, 4096, 4096, 4096, 1, 0, 0, 1, 1, 152) == 3
    assert ch(1, 1, 4096, 4096, 4096, 1, 0, 0, 1, 1, 152) == 2
    assert ch(1, 0, 4096, 4096, 4096, 1, 0, 0, 1, 1, 152) == 0
    assert ch(0, 1, 2048, 2048, 128, 128, 0, 0, 1, 1, 152) == 3
    assert ch(0, 0, 2048, 128, 2048, 128, 0, 0, 1, 1, 152) == 0
    assert ch(0, 0, 1024, 1024, 1024, 1, 0, 0, 1, 1, 152) == 0
    # an unaligned operand stored with k contiguous changes nothing (it is copied element
    # by element in any case): the same choices as aligned
    assert ch(0, 0, 1024, 1024, 1024, 1, 0, 0, 0, 1, 152) == 0
    assert ch(0, 0, 4096, 4096, 4096, 1, 0, 0, 0, 1, 152) == 1
    assert ch(0, 1, 2048, 2048, 128, 128, 0, 0, 0, 0, 152) == 3
    # an unaligned k-major operand: copying it (aligned rows) or both (a transpose of the
    # other) is the way to the 16-byte kernels for all but small problems; up to 256^3 the
    # element-wise kernel is as fast (measured 15.0 against about 14 us at 256^3)
    assert ch(0, 0, 1024, 1024, 1024, 1, 0, 0, 1, 0, 152) != 0
    assert ch(0, 0, 4096, 4096, 4096, 1, 0, 0, 0, 0, 152) == 3
    assert ch(1, 0, 4096, 4096, 4096, 1, 0, 0, 0, 1, 152) == 1  # A re-pitched
    assert ch(1, 0, 4096, 4096, 4096, 1, 0, 0, 1, 0, 152) == 2  # B re-pitched
    assert ch(0, 0, 256, 256, 256, 1, 0, 0, 1, 0, 152) == 0
    assert ch(0, 0, 64, 64, 64, 1, 0, 0, 0, 0, 152) == 0
    # a batch-shared operand is copied once: cheaper, so copied at least as readily
    assert ch(0, 0, 2048, 128, 2048, 128, 1, 0, 1, 1, 152) == 1
    # the workspace bounds the choice: 64 MiB holds the copy of A at 4096^3, not the
    # 128 MiB copies of Q or K of the QK^T batch
    assert ch(0, 0, 4096, 4096, 4096, 1, 0, 0, 1, 1, 152, 64 << 20) == 1
    assert ch(0, 0, 4096, 4096, 4096, 1, 0, 0, 1, 1, 152, (64 << 20) - 4) == 0
    assert ch(0, 1, 2048, 2048, 128, 128, 0, 0, 1, 1, 152, 64 << 20) == 0
    assert ch(0, 0, 4096, 4096, 4096, 1, 0, 0, 0, 0, 152, 0) == 0
    assert ch(0, 0, 0, 4, 4, 1, 0, 0, 1, 1, 152) == 0
    assert ch(0, 0, -1, 4, 4, 1, 0, 0, 1, 1, 152, 0) == -1
    assert ch(0, 0, 4, 4, 4, 1, 0, 0, 1, 1, 0, 1 << 20) == -1


@pytest.mark.parametrize("kw", [dict(stage=4), dict(stage=-2), dict(M=-1), dict(lda=1),
                                dict(workspace=FAKE + 4), dict(workspace=FAKE + 8, stage=0),
                                dict(workspace=0, stage=1), dict(workspace=0, stage=3),
                                dict(workspace_bytes=16, stage=2)])
def test_staged_validates_before_launch(kw):
    args = dict(ta=0, tb=1, M=64, N=64, K=64, lda=64, workspace=FAKE, stage=fg.STAGE_AUTO)
    args.update(kw)
    need = fg.staged_workspace_size(0, 1, 64, 64, 64, 1)
    wsb = args.get("workspace_bytes", need)
    st = fg.sgemm_staged(args["ta"], args["tb"], args["M"], args["N"], args["K"], 1.0, FAKE,
                         args["lda"], 0, FAKE, 64, 0, 0.0, FAKE, 64, 0, 1, None, False,
                         args["stage"], args["workspace"], wsb, check=False)
    assert st == fg.ERR_INVALID_VALUE


def test_max_dim_matches_the_header():
    text = open(HEADER, encoding="utf-8").read()
    m = re.search(r"#define\s+FGEMM_MAX_DIM\s+(\d+)", text)
    assert m and int(m.group(1)) == fg.MAX_DIM == 2**31 - 256


@pytest.mark.parametrize("dim", ["M", "N", "K"])
def test_sizes_above_the_limit_are_not_supported_before_launch(dim):
    # A valid call with one size past FGEMM_MAX_DIM is refused as not supported by every
    # entry point, before any CUDA call (the pointers are never dereferenced); at the
    # limit itself the size checks pass (the same calls then fail only on the missing
    # GPU or on the fake pointers, never with NOT_SUPPORTED from the size).  Invalid
    # arguments still come first, and an empty problem is still a no-op.
    over = fg.MAX_DIM + 1
    big = 2**31 - 1  # leading dimensions that cover any size
    base = dict(transa=0, transb=0, M=8, N=8, K=8, alpha=1.0, A=FAKE, lda=big, B=FAKE, ldb=big,
                beta=0.0, C=FAKE, ldc=big)
    kw = dict(base, **{dim: over})
    assert fg.sgemm(**kw, check=False) == fg.ERR_NOT_SUPPORTED
    assert fg.sgemm_bias_relu(**kw, bias=None, apply_relu=True, check=False) == fg.ERR_NOT_SUPPORTED
    assert fg.sgemm_row_bias_relu(**kw, row_bias=None, apply_relu=False,
                                  check=False) == fg.ERR_NOT_SUPPORTED
    a = (kw["transa"], kw["transb"], kw["M"], kw["N"], kw["K"], 1.0, FAKE, big, 0, FAKE, big, 0,
         0.0, FAKE, big, 0, 1)
    assert fg.sgemm_strided_batched(*a, check=False) == fg.ERR_NOT_SUPPORTED
    for config in (-1, 0, fg.num_configs() - 1):
        assert fg.gemm_explicit(config, *a, check=False) == fg.ERR_NOT_SUPPORTED
    for math in (fg.MATH_FP32, fg.MATH_TF32, fg.MATH_3XTF32):
        assert fg.gemm_math(math, *a, check=False) == fg.ERR_NOT_SUPPORTED
        assert fg.math_supported(math, *a[:12], 1) == (1 if math == fg.MATH_FP32 else 0)
    assert fg.sgemm_staged(*a, None, False, fg.STAGE_AUTO, None, 0,
                           check=False) == fg.ERR_NOT_SUPPORTED
    assert fg.sgemm_splitk(**kw, bias=None, apply_relu=False, splits=2, workspace=FAKE,
                           workspace_bytes=2**63, check=False) == fg.ERR_NOT_SUPPORTED
    assert fg.sgemm_splitk_noalloc(**kw, bias=None, apply_relu=False, splits=1,
                                   check=False) == fg.ERR_NOT_SUPPORTED
    # invalid before unsupported; empty before both
    assert fg.sgemm(**dict(kw, ldc=7), check=False) == fg.ERR_INVALID_VALUE
    assert fg.sgemm(**dict(kw, C=None), check=False) == fg.ERR_INVALID_VALUE
    empty = "N" if dim != "N" else "M"
    assert fg.sgemm(**dict(kw, **{empty: 0}), check=False) == fg.OK


@pytest.mark.parametrize("dim", ["M", "N", "K"])
def test_launch_count_at_and_above_the_limit(dim):
    # Host-only: sizes at the limit give a launch count from 64-bit tile arithmetic;
    # above it (refused as not supported) the call launches nothing.
    sizes = dict(M=8, N=8, K=8)
    for config in range(-1, fg.num_configs()):
        for ta in (0, 1):
            for tb in (0, 1):
                at = dict(sizes, **{dim: fg.MAX_DIM})
                n = fg.launch_count(config, ta, tb, at["M"], at["N"], at["K"], 1, 1, 152)
                assert 1 <= n <= 9, (config, ta, tb, n)
                above = dict(sizes, **{dim: fg.MAX_DIM + 1})
                assert fg.launch_count(config, ta, tb, above["M"], above["N"], above["K"], 1, 1,
                                       152) == 0


def test_launch_count_of_a_grid_too_large_for_one_launch():
    # 2^48 tiles of 128 x 128 exceed one grid: the launchers refuse the call as not
    # supported, so the query answers 0 (for TT whole tiles too, whose count divides by
    # the tiles a launch holds).
    side = fg.MAX_DIM
    for config in range(fg.num_configs()):
        assert fg.launch_count(config, 1, 1, side, side, 64, 1, 1, 152) == 0, config
        assert fg.launch_count(config, 0, 0, side, side, 64, 1, 1, 152) == 0, config
    # TT whole tiles: 2^31 - 256 tiles fill one launch (a batch of two takes two); one
    # more column of tiles is more than a launch holds
    assert fg.launch_count(0, 1, 1, fg.MAX_DIM, 128 * 128, 64, 1, 1, 152) == 1
    assert fg.launch_count(0, 1, 1, fg.MAX_DIM, 128 * 128, 64, 2, 1, 152) == 2
    assert fg.launch_count(0, 1, 1, fg.MAX_DIM, 128 * 128 + 1, 64, 1, 1, 152) == 0


def test_math_staged_workspace_size_and_choice():
    sz, ch = fg.math_staged_workspace_size, fg.math_staged_choice
    # K-major copies: A as M rows and B as N rows of ld4(K) floats a problem, B's at the
    # next multiple of 256 bytes
    for math in (fg.MATH_TF32, fg.MATH_3XTF32):
        assert sz(math, 1, 0, 4096, 4096, 4096, 1) == 2 * 4096 * 4096 * 4
        assert sz(math, 0, 0, 5, 7, 3, 2) == (2 * 5 * 4 * 4 + 255) // 256 * 256 + 2 * 7 * 4 * 4
        assert sz(math, 0, 0, 0, 7, 3, 1) == 0 and sz(math, 2, 0, 5, 7, 3, 1) == 0
    assert sz(fg.MATH_FP32, 0, 0, 5, 7, 3, 2) == fg.staged_workspace_size(0, 0, 5, 7, 3, 2)
    assert sz(7, 0, 0, 5, 7, 3, 2) == 0
    assert sz(fg.MATH_TF32, 0, 0, 2**31 - 1, 2**31 - 1, 2**31 - 1, 2**31 - 1) == 2**64 - 1
    for math in (fg.MATH_TF32, fg.MATH_3XTF32):
        # aligned operands: only TN is copied (A, so that it runs as NN)
        got = {(ta, tb): ch(math, ta, tb, 4096, 4096, 4096, 1, 0, 0, 1, 1, 152)
               for ta in (0, 1) for tb in (0, 1)}
        assert got == {(0, 0): 0, (0, 1): 0, (1, 0): 1, (1, 1): 0}
        # an unaligned operand is copied in any layout, two unaligned ones together
        assert all(ch(math, ta, tb, 512, 512, 512, 1, 0, 0, 0, 1, 152) == 1
                   for ta in (0, 1) for tb in (0, 1))
        assert all(ch(math, ta, tb, 512, 512, 512, 1, 0, 0, 1, 0, 152) == 2
                   for ta in (0, 1) for tb in (0, 1))
        assert ch(math, 0, 0, 512, 512, 512, 1, 0, 0, 0, 0, 152) == 3
        # within the workspace: TN falls back to B's copy when only it fits (N < M), two
        # unaligned operands are copied both or not at all, nothing without a workspace
        a_only = sz(math, 1, 0, 4096, 1024, 1024, 1) - 1024 * 1024 * 4
        assert ch(math, 1, 0, 4096, 1024, 1024, 1, 0, 0, 1, 1, 152, 1024 * 1024 * 4) == 2
        assert ch(math, 1, 0, 4096, 1024, 1024, 1, 0, 0, 1, 1, 152, a_only) == 1
        assert ch(math, 0, 0, 512, 512, 512, 1, 0, 0, 0, 0, 152, 512 * 512 * 4) == 0
        assert ch(math, 1, 0, 4096, 4096, 4096, 1, 0, 0, 1, 1, 152, 0) == 0
        # a batch that shares A copies it once
        one = ch(math, 1, 0, 256, 256, 256, 8, 1, 0, 1, 1, 152, 256 * 256 * 4)
        assert one == 1 and ch(math, 1, 0, 256, 256, 256, 8, 0, 0, 1, 1, 152, 256 * 256 * 4) == 0
    assert ch(fg.MATH_FP32, 0, 0, 4096, 4096, 4096, 1, 0, 0, 1, 1, 152) == \
        fg.staged_choice(0, 0, 4096, 4096, 4096, 1, 0, 0, 1, 1, 152)
    assert ch(7, 0, 0, 4, 4, 4, 1, 0, 0, 1, 1, 152) == -1
    assert ch(fg.MATH_TF32, 0, 0, -1, 4, 4, 1, 0, 0, 1, 1, 152) == -1


def test_math_staged_argument_checks_before_launch():
    M = N = K = 256
    args = (0, 0, M, N, K, 1.0, FAKE, K, 0, FAKE, N, 0, 0.0, FAKE, N, 0, 1, None, False)
    need_a = M * K * 4
    for math in (fg.MATH_TF32, fg.MATH_3XTF32):
        bad = [dict(stage=1, ws=None, wb=0), dict(stage=3, ws=FAKE, wb=need_a),
               dict(stage=-1, ws=FAKE + 4, wb=need_a), dict(stage=4, ws=FAKE, wb=need_a),
               dict(stage=-2, ws=FAKE, wb=need_a)]
        for kw in bad:
            assert fg.gemm_math_staged(math, *args, kw["stage"], kw["ws"], kw["wb"],
                                       check=False) == fg.ERR_INVALID_VALUE, kw
        bad_ld = (0, 0, M, N, K, 1.0, FAKE, K - 1, 0, FAKE, N, 0, 0.0, FAKE, N, 0, 1, None, False)
        assert fg.gemm_math_staged(math, *bad_ld, -1, None, 0, check=False) == fg.ERR_INVALID_VALUE
        empty = (0, 0, 0, N, K, 1.0, None, K, 0, None, N, 0, 0.0, None, N, 0, 1, None, False)
        assert fg.gemm_math_staged(math, *empty, -1, None, 0, check=False) == fg.OK
    assert fg.gemm_math_staged(5, *args, -1, None, 0, check=False) == fg.ERR_INVALID_VALUE
