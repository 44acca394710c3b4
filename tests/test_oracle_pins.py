"""The CPU oracle against facts fixed by the pages and the mathematics (no GPU)."""
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    assert pin(orc) is None
