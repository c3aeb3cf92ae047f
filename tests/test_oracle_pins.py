"""The CPU oracle against its pins (no GPU).  See ``tests/pins.py``."""
import pytest

import oracle
from tests import pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(lib, pin):
    pin(lib)


def test_rejects_nan_and_bad_args(lib):
    import numpy as np
    x = np.zeros((1, 4), dtype=np.uint16)
    x[0, 2] = 0x7FC0
    with pytest.raises(oracle.OracleError):
        oracle.topk(x, 2, lib=lib)
    with pytest.raises(oracle.OracleError):
        oracle.topk(np.zeros((1, 4), dtype=np.uint16), 5, lib=lib)
