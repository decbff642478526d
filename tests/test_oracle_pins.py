"""The CPU oracle against its pins (hand-worked values from the pages' format,
closed forms, invariants, brute force). No GPU needed."""
import pytest

from tests.oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()
