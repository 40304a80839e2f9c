"""The CPU oracle against its pins (hand-derived cases, closed forms,
brute force, library routines and the page's structural identities)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_mod):
    pin(oracle_mod.scan)


def test_oracle_rejects_bad_arguments(oracle_mod):
    import numpy as np
    x = np.zeros((2, 3, 4), np.float32)
    with pytest.raises(ValueError):       # NORMCAP needs a vector state
        oracle_mod.scan("NORMCAP", np.zeros((2, 4), np.float32), [x, x], axis=1)
    with pytest.raises(ValueError):       # initial of the wrong shape
        oracle_mod.scan("TANH_DECAY", np.zeros((2, 3), np.float32), [x, x], axis=1)
    with pytest.raises(ValueError):       # the state axis cannot be the scan axis
        oracle_mod.scan("NORMCAP", np.zeros((2, 3), np.float32), [x, x], axis=-1, state_axis=True)
    with pytest.raises(ValueError):       # axis out of range
        oracle_mod.scan("MAXPLUS", np.zeros((2, 4), np.float32), [x, x], axis=3)
