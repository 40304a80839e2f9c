"""The body-program oracle against its pins (no GPU)."""
import pytest

import body_pins
from oracle.body import scan_body


@pytest.mark.parametrize("pin", body_pins.ALL_PINS, ids=[p.__name__ for p in body_pins.ALL_PINS])
def test_body_pin(pin):
    pin(scan_body)
