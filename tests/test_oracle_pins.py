"""The float64 oracle against checks that do not use its arithmetic (tests/oracle_pins.py)."""
import pytest

import oracle
import oracle_pins as P


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(lib, pin):
    ok, detail = pin(lib)
    assert ok, detail
