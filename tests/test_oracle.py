"""The FP64 oracle against its pins (no GPU)."""

import numpy as np
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_rejects_bad_arguments(orc):
    A = np.ones(4, np.float32)
    with pytest.raises(ValueError):
        orc.gemm(2, 0, 2, 2, 2, 1.0, A, 2, A, 2)  # transpose flag out of range
    with pytest.raises(ValueError):
        orc.gemm(0, 0, 2, 2, 2, 1.0, A, 2, A, 2, rows=[2])  # row out of range
    with pytest.raises(ValueError):
        orc.gemm(0, 0, 2, 2, 2, 1.0, A, 2, A, 2, beta=1.0)  # beta != 0 needs C0


def test_empty_shapes(orc):
    out, mag = orc.gemm(0, 0, 0, 5, 3, 1.0, None, 3, np.ones(15, np.float32), 5)
    assert out.shape == (0, 5)
    out, mag = orc.gemm(0, 0, 4, 0, 3, 1.0, np.ones(12, np.float32), 3, None, 1)
    assert out.shape == (4, 0)
