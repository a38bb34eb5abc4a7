"""The oracle against what the definitions and the mathematics fix (CPU)."""
import pytest

from _pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__[4:])
def test_pin(pin, orc, kvalues):
    pin(orc, kvalues)
