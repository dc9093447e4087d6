"""Single problems whose C, A or B holds more than 2^31 elements.

Inside one problem the kernels address elements with 64-bit offsets, and tiles, rows,
columns and k with 32-bit positions (include/fgemm.h, "Sizes").  These cases put
element offsets past 2^31 in each array in turn -- the output, the operand read with k
contiguous, the operand read k-major -- through every kernel configuration, the last-wave
splits, the staged copies (transposed and re-pitched), split-K and the tensor cores.

An operand of 2^31 elements is too large to draw element by element for the oracle, so
it is built from a seeded pool of small-integer rows (workloads.pooled_ints): row r of
op(A) repeats pool row idx[r], column j of op(B) pool column jdx[j], and C's initial
values and the bias follow the same indices.  The FP64 oracle computes the pool's
products once (alpha, beta, bias and ReLU included); every product and sum is an
integer well inside FP32's exact range, so the WHOLE output must equal the oracle's
pool result gathered by the same indices, element by element and bit for bit.  Where
beta is 0, C starts as NaN, so an element the call does not write shows; padding
columns of C and of the operands hold NaN and must be neither written nor read.
"""

import numpy as np
import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
import oracle
from dense_fp32_gemm_sm_gb300 import workloads

pytestmark = pytest.mark.gpu

NAN = float("nan")
NUM_CONFIGS = 10  # fgemm_num_configs(); checked below
CHUNK = 1 << 18  # rows gathered per copy while building a large operand


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    fg.library()
    assert fg.num_configs() == NUM_CONFIGS
    if torch.cuda.mem_get_info()[0] < 48 * 2**30:
        pytest.skip("needs 48 GiB of free device memory")
    yield
    torch.cuda.empty_cache()


def _exact32(o: np.ndarray) -> torch.Tensor:
    """The oracle's FP64 result as FP32, checking that no value was rounded."""
    o32 = o.astype(np.float32)
    assert np.array_equal(o32.astype(np.float64), o), "the data must keep every value exact"
    return torch.from_numpy(o32)


def _rows_storage(pool_g, index_g, width, ld):
    """Rows pool_g[index_g[r]] (width floats each) in a device array with leading
    dimension ld; columns width .. ld-1 hold NaN."""
    n = index_g.numel()
    out = torch.full((n, ld), NAN, device="cuda")
    for r0 in range(0, n, CHUNK):
        r1 = min(r0 + CHUNK, n)
        out[r0:r1, :width] = pool_g[index_g[r0:r1]]
    return out


def _cols_storage(pool_g, index_g, width, ld):
    """The transpose: column c is pool_g[index_g[c]] (width rows), leading dimension ld;
    columns index_g.numel() .. ld-1 hold NaN."""
    n = index_g.numel()
    out = torch.full((width, ld), NAN, device="cuda")
    for c0 in range(0, n, CHUNK):
        c1 = min(c0 + CHUNK, n)
        out[:, c0:c1] = pool_g[index_g[c0:c1]].t()
    return out


def _workspace(nbytes):
    return torch.empty((nbytes + 3) // 4, device="cuda")


@pytest.fixture(scope="class")
def d(request):
    """The pools, indices and expected output of the class's case (its make_data)."""
    data = request.cls.make_data()
    yield data
    data.clear()
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------------
# C beyond 2^31 elements: 70001 x 32771 = 2,294,002,771 (K = 24, a single partial stage).


class TestOutputBeyond2to31:
    M, N, K, POOL = 70001, 32771, 24, 1024
    ALPHA = -0.5

    @classmethod
    def make_data(cls):
        g = workloads.generator(300)
        P, idx = workloads.pooled_ints(g, cls.M, cls.POOL, cls.K)  # rows of op(A)
        Qt, jdx = workloads.pooled_ints(g, cls.N, cls.POOL, cls.K)  # columns of op(B)
        o, _ = oracle.gemm(0, 1, cls.POOL, cls.POOL, cls.K, cls.ALPHA, P.numpy().reshape(-1),
                           cls.K, Qt.numpy().reshape(-1), cls.K, want_mag=False)
        idx_g, jdx_g = idx.cuda(), jdx.cuda()
        want = _exact32(o).cuda()[idx_g][:, jdx_g]
        assert (cls.M * cls.N) > 2**31 and want.shape == (cls.M, cls.N)
        return dict(P=P.cuda(), idx=idx_g, Qt=Qt.cuda(), jdx=jdx_g, want=want)

    def operands(self, d, ta, tb, lda_pad=0, ldb_pad=0):
        M, N, K = self.M, self.N, self.K
        if ta == 0:
            A, lda = _rows_storage(d["P"], d["idx"], K, K + lda_pad), K + lda_pad
        else:
            A, lda = _cols_storage(d["P"], d["idx"], K, M + lda_pad), M + lda_pad
        if tb == 1:
            B, ldb = _rows_storage(d["Qt"], d["jdx"], K, K + ldb_pad), K + ldb_pad
        else:
            B, ldb = _cols_storage(d["Qt"], d["jdx"], K, N + ldb_pad), N + ldb_pad
        return A, lda, B, ldb

    def check(self, d, C, ldc):
        torch.cuda.synchronize()
        assert torch.equal(C[:, :self.N], d["want"]), "an element differs from the oracle"
        if ldc > self.N:
            assert bool(torch.isnan(C[:, self.N:]).all()), "a padding column was written"

    @pytest.mark.parametrize("ldc_pad", [0, 1])
    @pytest.mark.parametrize("config", range(NUM_CONFIGS))
    def test_every_configuration(self, d, config, ldc_pad):
        # NN; ldc = N (odd: element stores) or N + 1 (16-byte stores)
        A, lda, B, ldb = self.operands(d, 0, 0, ldb_pad=1)
        ldc = self.N + ldc_pad
        C = torch.full((self.M, ldc), NAN, device="cuda")
        fg.gemm_explicit(config, 0, 0, self.M, self.N, self.K, self.ALPHA, A, lda, 0, B, ldb, 0,
                         0.0, C, ldc, 0, 1)
        self.check(d, C, ldc)

    @pytest.mark.parametrize("ta,tb", [(0, 1), (1, 0), (1, 1)])
    def test_other_layouts(self, d, ta, tb):
        A, lda, B, ldb = self.operands(d, ta, tb, lda_pad=3 if ta else 0, ldb_pad=0 if tb else 1)
        ldc = self.N + 1
        C = torch.full((self.M, ldc), NAN, device="cuda")
        fg.sgemm(ta, tb, self.M, self.N, self.K, self.ALPHA, A, lda, B, ldb, 0.0, C, ldc)
        self.check(d, C, ldc)

    @pytest.mark.parametrize("stage", [fg.STAGE_AUTO, 3])
    def test_staged(self, d, stage):
        A, lda, B, ldb = self.operands(d, 0, 1)
        need = fg.staged_workspace_size(0, 1, self.M, self.N, self.K, 1)
        ws = _workspace(need)
        ldc = self.N
        C = torch.full((self.M, ldc), NAN, device="cuda")
        fg.sgemm_staged(0, 1, self.M, self.N, self.K, self.ALPHA, A, lda, 0, B, ldb, 0, 0.0, C,
                        ldc, 0, 1, None, False, stage, ws, need)
        self.check(d, C, ldc)

    @pytest.mark.parametrize("math", [fg.MATH_TF32, fg.MATH_3XTF32])
    def test_tensor_cores(self, d, math):
        A, lda, B, ldb = self.operands(d, 0, 0, ldb_pad=1)
        assert fg.math_supported(math, 0, 0, self.M, self.N, self.K, self.ALPHA, A, lda, 0, B,
                                 ldb, 0, 1) == 1
        ldc = self.N + 1
        C = torch.full((self.M, ldc), NAN, device="cuda")
        fg.gemm_math(math, 0, 0, self.M, self.N, self.K, self.ALPHA, A, lda, 0, B, ldb, 0, 0.0,
                     C, ldc, 0, 1)
        self.check(d, C, ldc)
        assert fg.device_status() == fg.OK


# ---------------------------------------------------------------------------------
# An operand beyond 2^31 elements: op(A) 2097155 x 1029 (A stored with leading dimension
# 1032 or 2097156: 2,164,263,960 / 2,157,973,524 elements), or op(B) 1029 x 2097155; the
# other operand and C are small.  alpha = 2, beta = 0.5, bias and ReLU.


class _BigOperand:
    BIG, SMALL, K, POOL = 2097155, 36, 1029, 2048
    ALPHA, BETA = 2.0, 0.5

    def ws_for(self, ta, tb, M, N):
        need = fg.staged_workspace_size(ta, tb, M, N, self.K, 1)
        return _workspace(need), need


class TestOperandABeyond2to31(_BigOperand):
    @classmethod
    def make_data(cls):
        M, N, K = cls.BIG, cls.SMALL, cls.K
        g = workloads.generator(301)
        P, idx = workloads.pooled_ints(g, M, cls.POOL, K)  # rows of op(A)
        R = workloads.small_ints(g, (cls.POOL, N))  # rows of the initial C, by the same index
        B = workloads.small_ints(g, (K, N))  # op(B) = B, stored K x N
        bias = workloads.small_ints(g, (N,))
        o, _ = oracle.gemm(0, 0, cls.POOL, N, K, cls.ALPHA, P.numpy().reshape(-1), K,
                           B.numpy().reshape(-1), N, beta=cls.BETA, C0=R.numpy().reshape(-1),
                           ldc=N, bias=bias.numpy(), relu=True, want_mag=False)
        idx_g = idx.cuda()
        return dict(P=P.cuda(), idx=idx_g, B=B.cuda(), bias=bias.cuda(),
                    c0=R.cuda()[idx_g], want=_exact32(o).cuda()[idx_g])

    def a_storage(self, d, ta, aligned=True):
        if ta == 0:
            lda = self.K + 3
            return _rows_storage(d["P"], d["idx"], self.K, lda), lda
        lda = self.BIG + 1 if aligned else self.BIG
        return _cols_storage(d["P"], d["idx"], self.K, lda), lda

    def run(self, d, A, call):
        assert A.numel() > 2**31
        C = d["c0"].clone()
        call(C)
        torch.cuda.synchronize()
        assert torch.equal(C, d["want"]), "an element differs from the oracle"

    @pytest.mark.parametrize("config", range(NUM_CONFIGS))
    @pytest.mark.parametrize("ta", [0, 1])
    def test_every_configuration(self, d, ta, config):
        A, lda = self.a_storage(d, ta)
        M, N, K = self.BIG, self.SMALL, self.K
        self.run(d, A, lambda C: fg.gemm_explicit(
            config, ta, 0, M, N, K, self.ALPHA, A, lda, 0, d["B"], N, 0, self.BETA, C, N, 0, 1,
            bias=d["bias"], apply_relu=True))

    def test_unaligned_k_major(self, d):
        # op(A) = T with lda = M (odd): the element-copy configurations
        A, lda = self.a_storage(d, 1, aligned=False)
        M, N, K = self.BIG, self.SMALL, self.K
        self.run(d, A, lambda C: fg.sgemm_bias_relu(
            1, 0, M, N, K, self.ALPHA, A, lda, d["B"], N, self.BETA, C, N, d["bias"], True))

    @pytest.mark.parametrize("ta,aligned", [(0, True), (1, False)])
    def test_staged_copy(self, d, ta, aligned):
        # op(A) = N: A transposed into the workspace; op(A) = T unaligned: re-pitched
        A, lda = self.a_storage(d, ta, aligned)
        M, N, K = self.BIG, self.SMALL, self.K
        ws, need = self.ws_for(ta, 0, M, N)
        self.run(d, A, lambda C: fg.sgemm_staged(
            ta, 0, M, N, K, self.ALPHA, A, lda, 0, d["B"], N, 0, self.BETA, C, N, 0, 1, d["bias"],
            True, 1, ws, need))

    @pytest.mark.parametrize("ta", [0, 1])
    def test_split_k(self, d, ta):
        A, lda = self.a_storage(d, ta)
        M, N, K = self.BIG, self.SMALL, self.K
        need = fg.splitk_workspace_size(M, N, K, 3)
        ws = _workspace(need)
        self.run(d, A, lambda C: fg.sgemm_splitk(
            ta, 0, M, N, K, self.ALPHA, A, lda, d["B"], N, self.BETA, C, N, d["bias"], True, 3,
            ws, need))

    @pytest.mark.parametrize("math", [fg.MATH_TF32, fg.MATH_3XTF32])
    @pytest.mark.parametrize("ta", [0, 1])
    def test_tensor_cores(self, d, ta, math):
        A, lda = self.a_storage(d, ta)
        M, N, K = self.BIG, self.SMALL, self.K
        assert fg.math_supported(math, ta, 0, M, N, K, self.ALPHA, A, lda, 0, d["B"], N, 0, 1) == 1
        self.run(d, A, lambda C: fg.gemm_math(
            math, ta, 0, M, N, K, self.ALPHA, A, lda, 0, d["B"], N, 0, self.BETA, C, N, 0, 1,
            bias=d["bias"], apply_relu=True))
        assert fg.device_status() == fg.OK


class TestOperandBBeyond2to31(_BigOperand):
    @classmethod
    def make_data(cls):
        M, N, K = cls.SMALL, cls.BIG, cls.K
        g = workloads.generator(302)
        A = workloads.small_ints(g, (M, K))  # op(A) = A, stored M x K (leading dimension K + 3)
        Qt, jdx = workloads.pooled_ints(g, N, cls.POOL, K)  # columns of op(B)
        R = workloads.small_ints(g, (M, cls.POOL))  # columns of the initial C
        bias_pool = workloads.small_ints(g, (cls.POOL,))  # the bias, by the same index
        o, _ = oracle.gemm(0, 1, M, cls.POOL, K, cls.ALPHA, A.numpy().reshape(-1), K,
                           Qt.numpy().reshape(-1), K, beta=cls.BETA, C0=R.numpy().reshape(-1),
                           ldc=cls.POOL, bias=bias_pool.numpy(), relu=True, want_mag=False)
        jdx_g = jdx.cuda()
        A_st = torch.full((M, K + 3), NAN, device="cuda")
        A_st[:, :K] = A.cuda()
        return dict(A=A_st, Qt=Qt.cuda(), jdx=jdx_g, bias=bias_pool.cuda()[jdx_g],
                    c0=R.cuda()[:, jdx_g].contiguous(),
                    want=_exact32(o).cuda()[:, jdx_g].contiguous())

    def b_storage(self, d, tb, aligned=True):
        if tb == 1:
            ldb = self.K + 3
            return _rows_storage(d["Qt"], d["jdx"], self.K, ldb), ldb
        ldb = self.BIG + 1 if aligned else self.BIG
        return _cols_storage(d["Qt"], d["jdx"], self.K, ldb), ldb

    def run(self, d, B, call):
        assert B.numel() > 2**31
        C = d["c0"].clone()
        call(C)
        torch.cuda.synchronize()
        assert torch.equal(C, d["want"]), "an element differs from the oracle"

    @pytest.mark.parametrize("config", range(NUM_CONFIGS))
    @pytest.mark.parametrize("tb", [0, 1])
    def test_every_configuration(self, d, tb, config):
        B, ldb = self.b_storage(d, tb)
        M, N, K = self.SMALL, self.BIG, self.K
        self.run(d, B, lambda C: fg.gemm_explicit(
            config, 0, tb, M, N, K, self.ALPHA, d["A"], K + 3, 0, B, ldb, 0, self.BETA, C, N, 0, 1,
            bias=d["bias"], apply_relu=True))

    def test_unaligned_k_major(self, d):
        B, ldb = self.b_storage(d, 0, aligned=False)
        M, N, K = self.SMALL, self.BIG, self.K
        self.run(d, B, lambda C: fg.sgemm_bias_relu(
            0, 0, M, N, K, self.ALPHA, d["A"], K + 3, B, ldb, self.BETA, C, N, d["bias"], True))

    @pytest.mark.parametrize("tb,aligned", [(1, True), (0, False)])
    def test_staged_copy(self, d, tb, aligned):
        B, ldb = self.b_storage(d, tb, aligned)
        M, N, K = self.SMALL, self.BIG, self.K
        ws, need = self.ws_for(0, tb, M, N)
        self.run(d, B, lambda C: fg.sgemm_staged(
            0, tb, M, N, K, self.ALPHA, d["A"], K + 3, 0, B, ldb, 0, self.BETA, C, N, 0, 1, d["bias"],
            True, 2, ws, need))

    @pytest.mark.parametrize("tb", [0, 1])
    def test_split_k(self, d, tb):
        B, ldb = self.b_storage(d, tb)
        M, N, K = self.SMALL, self.BIG, self.K
        need = fg.splitk_workspace_size(M, N, K, 3)
        ws = _workspace(need)
        self.run(d, B, lambda C: fg.sgemm_splitk(
            0, tb, M, N, K, self.ALPHA, d["A"], K + 3, B, ldb, self.BETA, C, N, d["bias"], True, 3,
            ws, need))

    @pytest.mark.parametrize("math", [fg.MATH_TF32, fg.MATH_3XTF32])
    @pytest.mark.parametrize("tb", [0, 1])
    def test_tensor_cores(self, d, tb, math):
        B, ldb = self.b_storage(d, tb)
        M, N, K = self.SMALL, self.BIG, self.K
        assert fg.math_supported(math, 0, tb, M, N, K, self.ALPHA, d["A"], K + 3, 0, B, ldb, 0, 1) == 1
        self.run(d, B, lambda C: fg.gemm_math(
            math, 0, tb, M, N, K, self.ALPHA, d["A"], K + 3, 0, B, ldb, 0, self.BETA, C, N, 0, 1,
            bias=d["bias"], apply_relu=True))
        assert fg.device_status() == fg.OK
