"""The oracle's backward pass against its pins: central differences of the
f64 forward, PyTorch autograd of a plain loop (bit-exact for MAXPLUS, ties
included), a zero-decay closed form and the adjoint of the linear regime."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.BWD_PINS, ids=lambda f: f.__name__)
def test_backward_pin(pin, oracle_mod):
    pin(oracle_mod.scan, oracle_mod.scan_backward)
