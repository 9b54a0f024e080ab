"""The CPU oracle against what the pages and the mathematics fix (no GPU needed)."""

import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def o():
    return oracle.load()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(o, pin):
    pin(o)


def test_threads_reported(o):
    assert o.max_threads() >= 1
