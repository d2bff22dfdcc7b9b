"""The float64 oracle against facts fixed by the pages and the mathematics."""
import pytest

import oracle_pins as pins
from oracle import Oracle


@pytest.fixture(scope="module")
def orc():
    return Oracle()


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(orc, check):
    check(orc)
