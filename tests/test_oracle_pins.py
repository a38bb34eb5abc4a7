"""The oracle against what the definitions and the mathematics fix (CPU)."""
import pytest

from _pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__[4:])
def test_pin(pin, orc, kvalues):
    pin(orc, kvalues)


def test_roofline_gate_negative_control():
    """A call reported faster than HBM allows trips the gate; a plausible one
    does not (9.25 MB at 6.8 TB/s takes 1.36 us)."""
    from _gates import gate_roofline
    peak = 6.8e12
    assert gate_roofline(9.25e6, 1.36e-6 * 1.2, peak) is None
    assert gate_roofline(9.25e6, 1.36e-6 * 0.5, peak) is not None
    assert gate_roofline(9.25e6, 0.0, peak) is not None
