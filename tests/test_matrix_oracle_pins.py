"""The matrix-scan / linear-scan oracle against its pins (no GPU)."""
import pytest

import matrix_pins
import oracle.matrix as M


@pytest.mark.parametrize("pin", matrix_pins.ALL_PINS, ids=[p.__name__ for p in matrix_pins.ALL_PINS])
def test_matrix_pin(pin):
    pin(M)
