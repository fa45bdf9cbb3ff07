"""The oracle against facts the mathematics fixes (see ``pins.py``)."""

import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_rejects_bad_arguments(orc):
    import numpy as np
    A = np.ones((3, 4), dtype=np.float32)
    B = np.ones((5, 2), dtype=np.float32)
    with pytest.raises(ValueError):
        orc.sgemm(A, B)
    with pytest.raises(ValueError):
        orc.sgemm(A, np.ones((4, 2), dtype=np.float32), beta=1.0)   # C0 missing


def test_threads_reported(orc):
    assert orc.max_threads() >= 1
