"""The last-wave split launches against the FP64 oracle.

All compute the first (tiles - r) 128 x 128 tiles whole and then the last
r = tiles mod SMs another way: simt_128x128_t8x8_split as 64 x 64 quarter tiles
with four k-groups, simt_128x128_t8x8_ksplit as clusters of four CTAs that each
multiply one k-slice of a whole tile and add the partial sums through distributed
shared memory, simt_128x128_t8x8_kchain as S chained launches (S from 2 to 8, by the
launch-time model), one k-slice of every tile each, that add their products into C in
slice order.  These cases put whole and split tiles in one call, with split
tiles on the ragged bottom and right edges (quarters wholly outside the matrix are
skipped), on the last problem of a strided batch, with k-slices that are short or
empty, and in all four transpose layouts; integer data must come back bit-exact,
uniform data within 1e-5 * mag.
"""

import itertools

import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
from gpu_harness import Case, check

pytestmark = pytest.mark.gpu

COMBOS = list(itertools.product((0, 1), (0, 1)))


SPLITS = ["simt_128x128_t8x8_split", "simt_128x128_t8x8_ksplit", "simt_128x128_t8x8_kchain"]


def _config(name):
    ids = [i for i in range(fg.num_configs()) if fg.config_name(i) == name]
    assert len(ids) == 1
    return ids[0]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    fg.library()


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _tiles(M, N, batch=1):
    return -(-M // 128) * -(-N // 128) * batch


@pytest.mark.parametrize("split", SPLITS)
@pytest.mark.parametrize("ta,tb", COMBOS)
def test_whole_and_split_tiles_integer_exact(split, ta, tb):
    # 1700 x 1650: 14 x 13 = 182 tiles; the last ones include the bottom-right
    # corner tile (rows 1664..1699, columns 1536..1649).
    M, N, K = 1700, 1650, 70
    assert _tiles(M, N) % _sms() != 0
    check(Case(ta=ta, tb=tb, M=M, N=N, K=K, alpha=2.0, beta=-0.5, config=_config(split),
               pad=(4, 8, 4), seed=M + K + 2 * ta + tb))


@pytest.mark.parametrize("split", SPLITS)
@pytest.mark.parametrize("ta,tb", COMBOS)
def test_whole_and_split_tiles_uniform(split, ta, tb):
    M, N, K = 1500, 1800, 333
    check(Case(ta=ta, tb=tb, M=M, N=N, K=K, alpha=1.5, beta=0.5, ints=False, bias=True,
               relu=True, config=_config(split), seed=21 + 2 * ta + tb))


@pytest.mark.parametrize("split", SPLITS)
@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1)])
def test_split_tiles_on_the_last_problem_of_a_batch(split, ta, tb):
    # 5 problems of 8 x 8 tiles = 320 tiles: with about 150 SMs the quarter tiles
    # all come from the last problem.
    check(Case(ta=ta, tb=tb, M=1000, N=990, K=37, alpha=1.0, beta=1.0, batch=5,
               config=_config(split), seed=33 + tb))


@pytest.mark.parametrize("split", SPLITS)
def test_every_tile_split_when_fewer_tiles_than_sms(split):
    M, N = 700, 500
    assert _tiles(M, N) < _sms()
    for ta, tb in COMBOS:
        check(Case(ta=ta, tb=tb, M=M, N=N, K=150, alpha=-0.5, beta=2.0, bias=True,
                   config=_config(split), seed=40 + 2 * ta + tb))


@pytest.mark.parametrize("split", ["simt_128x128_t8x8_ksplit", "simt_128x128_t8x8_kchain"])
@pytest.mark.parametrize("K", [0, 1, 31, 32, 33, 97, 128, 129])
def test_k_slices_short_and_empty(split, K):
    # K slices are whole 32-deep stages: K <= 96 leaves the last slices empty.
    for ta, tb in COMBOS:
        check(Case(ta=ta, tb=tb, M=300, N=260, K=K, alpha=1.0, beta=0.5, bias=True, relu=True,
                   config=_config(split), seed=60 + K + 2 * ta + tb))


@pytest.mark.parametrize("ta,tb", COMBOS)
def test_kchain_beta_zero_never_reads_c(ta, tb):
    # beta = 0: the first slice writes alpha * P_0 without reading C (which holds NaN);
    # later slices read only what earlier slices wrote.  Row bias on the last slice.
    check(Case(ta=ta, tb=tb, M=1900, N=1700, K=300, alpha=1.0, beta=0.0, c_nan=True, bias=True,
               relu=True, config=_config("simt_128x128_t8x8_kchain"), pad=(4, 8, 4),
               seed=70 + 2 * ta + tb))
    check(Case(ta=ta, tb=tb, M=1900, N=1700, K=300, alpha=-1.0, beta=0.0, c_nan=True,
               ints=False, config=_config("simt_128x128_t8x8_kchain"), seed=75 + 2 * ta + tb))


@pytest.mark.parametrize("slices", range(2, 9))
def test_kchain_every_slice_count(slices):
    # The k-chain cuts the last wave into 2 to 8 k-slices, as many as the launch-time
    # model finds fastest for the wave's size and K; fgemm_launch_count reports the
    # choice (one whole-tile launch, then one launch per slice).  The smallest ragged
    # shape with whole tiles that takes this many slices, in one of the four layouts.
    sms = _sms()
    cfg = _config("simt_128x128_t8x8_kchain")
    ta, tb = COMBOS[slices % 4]
    best = None
    for K in (96, 256, 512, 1024, 1536, 2048, 3072, 4096, 6144, 8192):
        for mt in range(10, 21):
            for nt in range(10, 21):
                M, N = 128 * mt - 37, 128 * nt - 5
                if mt * nt > sms and fg.launch_count(cfg, ta, tb, M, N, K, 1, True,
                                                     sms) == 1 + slices:
                    if best is None or M * N * K < best[0]:
                        best = (M * N * K, M, N, K)
    if best is None:
        assert sms != 152, "no shape takes %d slices on 152 SMs" % slices
        pytest.skip("no shape in the search takes %d slices on %d SMs" % (slices, sms))
    _, M, N, K = best
    check(Case(ta=ta, tb=tb, M=M, N=N, K=K, alpha=1.5, beta=-0.5, bias=True,
               relu=slices % 2 == 0, ints=slices % 2 == 1, config=cfg, pad=(4, 8, 4),
               seed=80 + slices))


@pytest.mark.parametrize("split", SPLITS)
def test_no_remainder_runs_whole_tiles_only(split):
    sms = _sms()
    M, N = 128 * sms, 256  # exactly 2 * SMs tiles
    check(Case(M=M, N=N, K=24, alpha=1.0, beta=0.0, config=_config(split), seed=50))


def test_selector_on_this_gpu():
    # The workloads whose remainder of tiles is small enough take the split on a
    # 152-SM GB300; the others keep whole tiles.
    sms = _sms()
    if sms != 152:
        pytest.skip("expectations measured on 152 SMs")
    name = lambda *a: fg.config_name(fg.select_config(*a, True, sms))
    assert name(0, 0, 4096, 4096, 4096, 1) == "simt_128x128_t8x8_kchain"
    assert name(0, 0, 8192, 11008, 4096, 1) == "simt_128x128_t8x8_ksplit"
    assert name(0, 0, 2048, 128, 2048, 128) == "simt_128x128_t8x8_ksplit"
    assert name(0, 1, 2048, 2048, 128, 128) == "simt_128x128_t8x8"
    assert name(0, 0, 3072, 3072, 3072, 1) == "simt_128x128_t8x8_kchain"
