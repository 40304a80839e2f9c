"""The table-scan oracle against its pins, and planted mistakes (no GPU)."""
import importlib.util
import os

import pytest

import table_pins
import oracle.table as TS

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "table.py")


@pytest.mark.parametrize("pin", table_pins.ALL_PINS, ids=[p.__name__ for p in table_pins.ALL_PINS])
def test_table_pin(pin):
    pin(TS)


MUTATIONS = [
    ("operands_swapped", "nxt = table[h, s].astype(np.int64)", "nxt = table[np.clip(s, 0, n_states - 1), np.clip(h, 0, n_syms - 1)].astype(np.int64)"),
    ("start_ignored", "h = np.full(sym.shape[0], start, dtype=np.int64)", "h = np.zeros(sym.shape[0], dtype=np.int64)"),
    ("state_not_clamped", "            nxt = np.clip(nxt, 0, n_states - 1)", "            nxt = nxt % n_states"),
    ("symbol_wraps", "            s = np.clip(s, 0, n_syms - 1)", "            s = s % n_syms"),
    ("previous_state_stored", "        h = nxt\n        out[:, t] = h", "        out[:, t] = h\n        h = nxt"),
    ("axis_ignored", "sym = np.moveaxis(symbols, ax, -1)", "sym = np.moveaxis(symbols, -1, -1)"),
    ("start_range_unchecked", "if not 0 <= start < n_states:", "if False:"),
]


@pytest.mark.parametrize("mid,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_table_pins_catch_mutant(mid, old, new, tmp_path):
    src = open(SRC).read()
    assert old in src, mid
    path = tmp_path / ("table_%s.py" % mid)
    path.write_text(src.replace(old, new, 1))
    spec = importlib.util.spec_from_file_location("table_mutant_%s" % mid, str(path))
    mutant = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mutant)
    caught = []
    for pin in table_pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError, IndexError):   # noqa: PERF203
            caught.append(pin.__name__)
    assert caught, "no table pin caught the planted mistake %s" % mid
