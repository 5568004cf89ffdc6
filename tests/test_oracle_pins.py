"""The CPU oracle against the facts that pin it (see oracle_pins.py)."""
import pytest

from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(pin, oracle_lib):
    pin(oracle_lib, quick=False)
