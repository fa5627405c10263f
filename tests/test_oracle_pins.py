"""The CPU oracle against its pins (closed forms, invariants, finite differences,
brute force, hand-worked page examples and float64 library routines)."""
import pytest

from oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()
