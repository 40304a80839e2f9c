"""The body-program gradient oracle against its pins, and planted mistakes
in a copy of it (no GPU)."""
import importlib.util
import os
import sys

import pytest

import body_grad_pins
from oracle.body import scan_body
from oracle.body_grad import scan_body_backward

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "body_grad.py")


@pytest.mark.parametrize("pin", body_grad_pins.ALL_PINS, ids=[p.__name__ for p in body_grad_pins.ALL_PINS])
def test_body_grad_pin(pin):
    pin(scan_body, scan_body_backward)


MUTATIONS = [
    ("sub_second_sign", 'return [(a, g), (b, np.negative(g))]', 'return [(a, g), (b, g)]'),
    ("mul_operands_swapped", 'return [(a, _fmul(g, b.v)), (b, _fmul(g, a.v))]',
     'return [(a, _fmul(g, a.v)), (b, _fmul(g, b.v))]'),
    ("div_denominator_sign", 'return [(a, _fdiv(g, b.v)), (b, np.negative(_fdiv(_fmul(g, out), b.v)))]',
     'return [(a, _fdiv(g, b.v)), (b, _fdiv(_fmul(g, out), b.v))]'),
    ("tanh_derivative", 'return [(a, _fmul(g, _fsub(f32(1.0), _fmul(out, out))))]',
     'return [(a, _fmul(g, _fadd(f32(1.0), _fmul(out, out))))]'),
    ("sqrt_factor", 'return [(a, _fdiv(_fmul(g, f32(0.5)), out))]', 'return [(a, _fdiv(g, out))]'),
    ("where_branches_swapped", 'return [(a, np.where(m, g, zero)), (b, np.where(m, zero, g))]',
     'return [(a, np.where(m, zero, g)), (b, np.where(m, g, zero))]'),
    ("maximum_tie_not_split", 'ga = np.where(a_wins, g, np.where(b_wins, zero, half))',
     'ga = np.where(a_wins, g, np.where(b_wins, zero, g))'),
    ("rmax_count_ignored", 'return [(a, np.where(eq, _fdiv(np.broadcast_to(g, a.v.shape), count), zero))]',
     'return [(a, np.where(eq, np.broadcast_to(g, a.v.shape), zero))]'),
    ("narrow_not_summed", '        c = _sum_w(c)                     # a width-one operand of a wide operation',
     '        c = c[:, 0:1]'),
    ("accumulate_overwrites", 'grads[operand.idx] = c if prev is None else _fadd(prev, c)',
     'grads[operand.idx] = c'),
    ("carried_cotangent_dropped", '        lam = _fadd(lam, gv[:, t].reshape(lanes, W))',
     '        lam = gv[:, t].reshape(lanes, W)'),
    ("wrong_direction", '    order = range(T) if reverse else range(T - 1, -1, -1)',
     '    order = range(T - 1, -1, -1) if reverse else range(T)'),
    ("previous_state_is_own", '        tp = t + 1 if reverse else t - 1', '        tp = t'),
    ("atan2_x_sign", 'return [(a, _fdiv(_fmul(g, b.v), den)), (b, np.negative(_fdiv(_fmul(g, a.v), den)))]',
     'return [(a, _fdiv(_fmul(g, b.v), den)), (b, _fdiv(_fmul(g, a.v), den))]'),
    ("cos_sign", 'return [(a, np.negative(_fmul(g, _via_f64(np.sin, a.v))))]',
     'return [(a, _fmul(g, _via_f64(np.sin, a.v)))]'),
]


@pytest.mark.parametrize("mid,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_body_grad_pins_catch_mutant(mid, old, new, tmp_path):
    src = open(SRC).read()
    assert old in src, mid
    pkg = tmp_path / "oracle"
    pkg.mkdir()
    root = os.path.dirname(SRC)
    for name in ("__init__.py", "body.py", "es_oracle.c"):
        (pkg / name).write_text(open(os.path.join(root, name)).read())
    (pkg / "body_grad.py").write_text(src.replace(old, new, 1))
    spec = importlib.util.spec_from_file_location("oracle_mut_%s.body_grad" % mid, str(pkg / "body_grad.py"),
                                                  submodule_search_locations=None)
    # load the copy as a submodule of a throwaway package so its relative import finds body.py
    pspec = importlib.util.spec_from_file_location("oracle_mut_%s" % mid, str(pkg / "__init__.py"),
                                                   submodule_search_locations=[str(pkg)])
    parent = importlib.util.module_from_spec(pspec)
    sys.modules["oracle_mut_%s" % mid] = parent
    pspec.loader.exec_module(parent)
    mutant = importlib.util.module_from_spec(spec)
    sys.modules["oracle_mut_%s.body_grad" % mid] = mutant
    spec.loader.exec_module(mutant)
    caught = []
    for pin in body_grad_pins.ALL_PINS:
        if pin is body_grad_pins.pin_tape_forward:
            continue
        try:
            pin(scan_body, mutant.scan_body_backward)
        except (AssertionError, ValueError):   # noqa: PERF203
            caught.append(pin.__name__)
    assert caught, "no gradient pin caught the planted mistake %s" % mid
