"""The oracle's sampled verify against its pins (no GPU).  See
``tests/pins_sampled.py``."""
import pytest

import oracle
from tests import pins_sampled


@pytest.fixture(scope="module", autouse=True)
def _lib():
    oracle.load()


@pytest.mark.parametrize("pin", pins_sampled.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle)
