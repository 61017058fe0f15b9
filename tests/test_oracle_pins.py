"""The CPU oracle against what the page and the mathematics fix (see
tests/oracle_pins.py for what each pin rests on)."""
import pytest

from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=[p.__name__ for p in ALL_PINS])
def test_pin(orc, pin):
    pin(orc)
