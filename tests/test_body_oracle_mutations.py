"""Plant plausible mistakes in the body-program oracle (a temporary copy of its
source, on the CPU) and check that the body pins catch every one of them.
The committed oracle is never touched."""
import importlib.util
import os

import pytest

import body_pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "body.py")

# (id, text in the interpreter, replacement, which occurrence (0-based))
MUTATIONS = [
    ("sub_operands_swapped", "np.subtract(a, b, dtype=np.float32)", "np.subtract(b, a, dtype=np.float32)", 0),
    ("add_as_sub", "np.add(a, b, dtype=np.float32)", "np.subtract(a, b, dtype=np.float32)", 0),
    ("div_operands_swapped", "np.divide(a, b, dtype=np.float32)", "np.divide(b, a, dtype=np.float32)", 0),
    ("greater_as_greater_equal", '">": np.greater,', '">": np.greater_equal,', 0),
    ("less_as_less_equal", '"<": np.less,', '"<": np.less_equal,', 0),
    ("not_equal_as_equal", '"!=": np.not_equal,', '"!=": np.equal,', 0),
    ("where_branches_swapped", "return np.where(m, a, b)", "return np.where(m, b, a)", 0),
    ("sum_drops_last_value", "for w in range(1, t.shape[1]):", "for w in range(1, t.shape[1] - 1):", 0),
    ("sum_in_reverse_order", "acc = t[:, 0:1]\n    for w in range(1, t.shape[1]):",
     "acc = t[:, -1:]\n    for w in range(t.shape[1] - 2, -1, -1):", 0),
    ("max_reduction_is_minimum", "else _ieee_maximum(acc, t[:, w:w + 1])", "else _ieee_minimum(acc, t[:, w:w + 1])",
     0),
    ("maximum_zero_sign", "eq = np.where(np.signbit(a), b, a)", "eq = a", 0),
    ("minimum_drops_nan", "return np.where(nan, np.float32(np.nan), r).astype(np.float32)",
     "return r.astype(np.float32)", 1),
    ("reverse_ignored", "order = range(T - 1, -1, -1) if reverse else range(T)", "order = range(T)", 0),
    ("let_binds_in_parallel", "inner[b[0]] = _eval(b[1], inner, ctx)", "inner[b[0]] = _eval(b[1], env, ctx)", 0),
    ("bool_cast_is_positive", "(v != np.float32(0))", "(v > np.float32(0))", 0),
    ("numbers_not_folded", "if _is_num(acc) and _is_num(v):", "if False:", 0),
    ("atan2_operands_swapped", "_via_f64(np.arctan2, a, b)", "_via_f64(np.arctan2, b, a)", 0),
    ("rsqrt_is_sqrt", '"rsqrt": lambda v: 1.0 / np.sqrt(v),', '"rsqrt": lambda v: np.sqrt(v),', 0),
    ("pow_operands_swapped", "_via_f64(np.power, a, b)", "_via_f64(np.power, b, a)", 0),
    ("exp_is_expm1", '"exp": np.exp,', '"exp": np.expm1,', 0),
    ("log_is_log1p", '"log": np.log,', '"log": np.log1p,', 0),
    ("initial_ignored", "h = initial.reshape(lanes, W).copy()", "h = np.zeros((lanes, W), np.float32)", 0),
    ("sequence_time_shift", "vals = [v[:, t].reshape(lanes, w)", "vals = [v[:, (t + 1) % T].reshape(lanes, w)", 0),
    ("and_is_or", 'acc = (acc & t) if head == "and" else (acc | t)', "acc = acc | t", 0),
    ("not_ignored", 'return ~_bool(vals[0], L, "not")', 'return _bool(vals[0], L, "not")', 0),
    ("unary_minus_ignored", 'if head == "-":\n                return np.negative(t)',
     'if head == "-":\n                return t', 0),
    ("unbound_name_reads_zero",
     'raise BodyError("E-SCAN-001", "`%s` is not an argument of the body or a let binding" % form)', "return 0.0", 0),
    ("scalar_state_may_reduce", "if not ctx.vector:\n        raise BodyError(\"reduce\"",
     "if False:\n        raise BodyError(\"reduce\"", 0),
    ("gate_not_broadcast", "if head == \"broadcast-to\" and len(dims) >= 1", "if False and len(dims) >= 1", 0),
]


def _mutate(src, old, new, occ):
    idx = -1
    for _ in range(occ + 1):
        idx = src.index(old, idx + 1)
    return src[:idx] + new + src[idx + len(old):]


def test_mutation_targets_exist():
    src = open(SRC).read()
    for mid, old, new, occ in MUTATIONS:
        assert src.count(old) > occ, mid


@pytest.mark.parametrize("mid,old,new,occ", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_body_pins_catch_mutant(mid, old, new, occ, tmp_path):
    src = open(SRC).read()
    mutated = _mutate(src, old, new, occ)
    assert mutated != src
    path = tmp_path / ("body_%s.py" % mid)
    path.write_text(mutated)
    spec = importlib.util.spec_from_file_location("body_mutant_%s" % mid, str(path))
    mutant = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mutant)
    caught = []
    for pin in body_pins.ALL_PINS:
        try:
            pin(mutant.scan_body)
        except (AssertionError, ValueError):   # noqa: PERF203
            caught.append(pin.__name__)
    assert caught, "no body pin caught the planted mistake %s" % mid
