"""Seeded random cases across the whole argument space, against the FP64 oracle.

Each case draws a transpose combination, ragged M, N, K, alpha/beta from values that
keep integer arithmetic exact, the epilogue options, a strided batch, padded leading
dimensions, unaligned pointers, an explicit kernel configuration or the library's own
choice, and the arithmetic (CUDA cores, TF32, 3xTF32); further cases go through the
staged entry with a random staging mask, shared batch operands and any alignment.
Integer-valued data makes every case bit-exact, so any dropped, duplicated or misplaced
partial product shows.
"""

import random

import pytest
import torch

import dense_fp32_gemm_sm_gb300 as fg
from gpu_harness import Case, check

pytestmark = pytest.mark.gpu

N_CASES = 96


def draw(rng):
    kw = dict(ta=rng.randint(0, 1), tb=rng.randint(0, 1), M=rng.randint(1, 320),
              N=rng.randint(1, 320), K=rng.choice([0, 1, 7, 16, 33, rng.randint(1, 320)]),
              alpha=rng.choice([1.0, 2.0, -0.5]), beta=rng.choice([0.0, 1.0, -2.0]),
              bias=rng.random() < 0.5, relu=rng.random() < 0.5,
              batch=rng.choice([0, 0, 1, 2, 3]),
              pad=(rng.choice([0, 1, 4]), rng.choice([0, 3, 8]), rng.choice([0, 2, 4])),
              seed=rng.randint(0, 1 << 30))
    unaligned = rng.random() < 0.25
    if unaligned:
        kw.update(offset=(rng.randint(0, 3), rng.randint(0, 3), rng.randint(0, 3)), align_ld=False)
    kw["c_nan"] = kw["beta"] == 0.0 and rng.random() < 0.5
    path = rng.random()
    if kw["batch"] and kw["bias"]:
        kw["bias"] = False  # the strided-batch entry point has no epilogue options
    if path < 0.3:
        kw["math"] = rng.choice([fg.MATH_TF32, fg.MATH_3XTF32])
        kw["expect_tc"] = None  # random offsets and padding decide the path
    elif path < 0.7 and not unaligned:
        kw["config"] = rng.randrange(fg.num_configs())
    return kw


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case(i):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    check(Case(**draw(random.Random(1000 + i))))


N_SPLIT_CASES = 24
SPLITS = ("simt_128x128_t8x8_split", "simt_128x128_t8x8_ksplit", "simt_128x128_t8x8_kchain")


def draw_split(rng):
    # grids larger than the SM count, so that whole tiles and a last wave of split
    # tiles (quarters, k-slice clusters or chained k-slices) meet in one call, on
    # ragged edges
    kw = dict(ta=rng.randint(0, 1), tb=rng.randint(0, 1), M=rng.randint(1500, 2600),
              N=rng.randint(1500, 2600), K=rng.choice([1, 31, 64, 97, rng.randint(1, 200)]),
              alpha=rng.choice([1.0, 2.0, -0.5]), beta=rng.choice([0.0, 1.0, -2.0]),
              bias=rng.random() < 0.5, relu=rng.random() < 0.5,
              batch=rng.choice([0, 0, 2]),
              pad=(rng.choice([0, 4]), rng.choice([0, 8]), rng.choice([0, 4])),
              seed=rng.randint(0, 1 << 30))
    if kw["batch"]:
        kw["bias"] = False
    name = rng.choice(SPLITS)
    kw["config"] = [i for i in range(fg.num_configs()) if fg.config_name(i) == name][0]
    return kw


@pytest.mark.parametrize("i", range(N_SPLIT_CASES))
def test_random_split_case(i):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    check(Case(**draw_split(random.Random(5000 + i))))


N_STAGED_CASES = 40


def draw_staged(rng):
    # fgemm_sgemm_staged: a random staging mask (or the model's choice) over the whole
    # argument space, with bias and ReLU on batches and operands a batch shares
    kw = dict(ta=rng.randint(0, 1), tb=rng.randint(0, 1), M=rng.randint(1, 700),
              N=rng.randint(1, 700), K=rng.choice([0, 1, 5, 32, 65, rng.randint(1, 400)]),
              alpha=rng.choice([1.0, 2.0, -0.5, 0.0]), beta=rng.choice([0.0, 1.0, -2.0]),
              bias=rng.random() < 0.5, relu=rng.random() < 0.5,
              batch=rng.choice([0, 0, 1, 3, 5]),
              pad=(rng.choice([0, 1, 4]), rng.choice([0, 3, 8]), rng.choice([0, 2, 4])),
              stage=rng.choice([fg.STAGE_AUTO, 0, 1, 2, 3]), seed=rng.randint(0, 1 << 30))
    if rng.random() < 0.3:
        kw.update(offset=(rng.randint(0, 3), rng.randint(0, 3), rng.randint(0, 3)), align_ld=False)
    if kw["batch"] > 1:
        kw["share_a"] = rng.random() < 0.3
        kw["share_b"] = rng.random() < 0.3
    kw["c_nan"] = kw["beta"] == 0.0 and rng.random() < 0.5
    return kw


@pytest.mark.parametrize("i", range(N_STAGED_CASES))
def test_random_staged_case(i):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    check(Case(**draw_staged(random.Random(9000 + i))))
