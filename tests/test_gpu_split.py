"""The last-wave split launch (simt_128x128_t8x8_split) against the FP64 oracle.

The split launch computes the first (tiles - r) 128 x 128 tiles whole and the
last r = tiles mod SMs as 64 x 64 quarter tiles with four k-groups.  These cases
put whole and quarter tiles in one launch, with the quarter tiles on the ragged
bottom and right edges (quarters wholly outside the matrix are skipped), on the
last problem of a strided batch, and in all four transpose layouts; integer data
must come back bit-exact, uniform data within 1e-5 * mag.
"""

import itertools

import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
from gpu_harness import Case, check

pytestmark = pytest.mark.gpu

COMBOS = list(itertools.product((0, 1), (0, 1)))


def _split_config():
    ids = [i for i in range(fg.num_configs()) if fg.config_name(i) == "simt_128x128_t8x8_split"]
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


@pytest.mark.parametrize("ta,tb", COMBOS)
def test_whole_and_quarter_tiles_integer_exact(ta, tb):
    # 1700 x 1650: 14 x 13 = 182 tiles; the last ones include the bottom-right
    # corner tile (rows 1664..1699, columns 1536..1649).
    M, N, K = 1700, 1650, 70
    assert _tiles(M, N) % _sms() != 0
    check(Case(ta=ta, tb=tb, M=M, N=N, K=K, alpha=2.0, beta=-0.5, config=_split_config(),
               pad=(4, 8, 4), seed=M + K + 2 * ta + tb))


@pytest.mark.parametrize("ta,tb", COMBOS)
def test_whole_and_quarter_tiles_uniform(ta, tb):
    M, N, K = 1500, 1800, 333
    check(Case(ta=ta, tb=tb, M=M, N=N, K=K, alpha=1.5, beta=0.5, ints=False, bias=True,
               relu=True, config=_split_config(), seed=21 + 2 * ta + tb))


@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1)])
def test_quarter_tiles_on_the_last_problem_of_a_batch(ta, tb):
    # 5 problems of 8 x 8 tiles = 320 tiles: with about 150 SMs the quarter tiles
    # all come from the last problem.
    check(Case(ta=ta, tb=tb, M=1000, N=990, K=37, alpha=1.0, beta=1.0, batch=5,
               config=_split_config(), seed=33 + tb))


def test_all_tiles_quartered_when_fewer_tiles_than_sms():
    M, N = 700, 500
    assert _tiles(M, N) < _sms()
    for ta, tb in COMBOS:
        check(Case(ta=ta, tb=tb, M=M, N=N, K=150, alpha=-0.5, beta=2.0, bias=True,
                   config=_split_config(), seed=40 + 2 * ta + tb))


def test_no_remainder_runs_whole_tiles_only():
    sms = _sms()
    M, N = 128 * sms, 256  # exactly 2 * SMs tiles
    check(Case(M=M, N=N, K=24, alpha=1.0, beta=0.0, config=_split_config(), seed=50))


def test_selector_on_this_gpu():
    # The workloads whose remainder of tiles is small enough take the split on a
    # 152-SM GB300; the others keep whole tiles.
    sms = _sms()
    if sms != 152:
        pytest.skip("expectations measured on 152 SMs")
    name = lambda *a: fg.config_name(fg.select_config(*a, True, sms))
    assert name(0, 0, 4096, 4096, 4096, 1) == "simt_128x128_t8x8_split"
    assert name(0, 0, 8192, 11008, 4096, 1) == "simt_128x128_t8x8_split"
    assert name(0, 0, 2048, 128, 2048, 128) == "simt_128x128_t8x8_split"
    assert name(0, 1, 2048, 2048, 128, 128) == "simt_128x128_t8x8"
    assert name(0, 0, 3072, 3072, 3072, 1) == "simt_128x128_t8x8"
