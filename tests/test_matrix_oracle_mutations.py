"""Plant plausible mistakes in the matrix-scan oracle (a temporary copy of its
source, on the CPU) and check that the pins catch every one of them."""
import importlib.util
import os

import pytest

import matrix_pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "matrix.py")

# (id, text in the oracle, replacement, which occurrence (0-based))
MUTATIONS = [
    ("transposed_a", "acc = np.multiply(a[:, :, 0:1], h[:, 0:1, :], dtype=np.float32)",
     "a = np.swapaxes(a, 1, 2)\n    acc = np.multiply(a[:, :, 0:1], h[:, 0:1, :], dtype=np.float32)", 0),
    ("last_term_dropped", "for j in range(1, n):", "for j in range(1, n - 1 if n > 1 else 1):", 0),
    ("b_dropped", "h = np.add(_product(at, h), bm[t], dtype=np.float32)", "h = _product(at, h)", 0),
    ("b_before_product", "h = np.add(_product(at, h), bm[t], dtype=np.float32)",
     "h = _product(at, np.add(h, bm[t], dtype=np.float32))", 0),
    ("h_starts_at_one", "h = np.zeros((L, n, m), np.float32)", "h = np.ones((L, n, m), np.float32)", 0),
    ("reverse_ignored", "order = range(T - 1, -1, -1) if reverse else range(T)", "order = range(T)", 0),
    ("projective_divides_before_b", "                h = np.divide(h, s, dtype=np.float32)",
     "                h = np.divide(np.subtract(h, bm[t], dtype=np.float32), s, dtype=np.float32) + bm[t]", 0),
    ("projective_max_without_abs", "s = np.abs(P).reshape(L, -1).max(axis=1)", "s = P.reshape(L, -1).max(axis=1)", 0),
    ("projective_product_not_carried", "                P = _product(at, P)",
     "                P = _product(at, np.broadcast_to(np.eye(n, dtype=np.float32), (L, n, n)))", 0),
    ("projective_h_not_scaled", "                h = np.divide(h, s, dtype=np.float32)", "                pass", 0),
    ("time_shift", "at = np.ascontiguousarray(am[t])", "at = np.ascontiguousarray(am[(t + 1) % T])", 0),
    ("broadcast_to_first_lane", "a = np.broadcast_to(a, lead + (n, n))",
     "a = np.broadcast_to(a.reshape((-1, n, n))[:1].reshape((1,) * len(lead) + (n, n)), lead + (n, n))", 0),
    ("n_limit_dropped", "if n > 16:", "if n > 64:", 0),
    ("bwd_not_transposed", "aT = np.ascontiguousarray(np.swapaxes(am[tn], 1, 2)) if 0 <= tn < T else zero_a",
     "aT = np.ascontiguousarray(am[tn]) if 0 <= tn < T else zero_a", 0),
    ("bwd_a_not_shifted", "tn = t - 1 if reverse else t + 1", "tn = t", 0),
    ("bwd_g_scaled", "lam = np.add(_product(aT, lam), gm[t], dtype=np.float32)",
     "lam = np.add(_product(aT, lam), gm[t] * np.float32(0.5), dtype=np.float32)", 0),
    ("bwd_h_not_previous", "tp = t + 1 if reverse else t - 1", "tp = t", 0),
    ("bwd_da_transposed", "da[t] = _outer_sum(lam, hp)", "da[t] = np.swapaxes(_outer_sum(lam, hp), 1, 2)", 0),
    ("bwd_wrong_direction", "order = range(T) if reverse else range(T - 1, -1, -1)",
     "order = range(T - 1, -1, -1) if reverse else range(T)", 0),
    ("bwd_projective_allowed", "    if projective:\n        raise", "    if False:\n        raise", 0),
    ("bwd_last_k_dropped", "for k in range(1, m):", "for k in range(1, m - 1 if m > 1 else 1):", 0),
    ("linear_scan_swapped", "r = matrix_scan(np.broadcast_to(a, shape)[..., None, None], np.broadcast_to(b, shape)[..., None, None],",
     "r = matrix_scan(np.broadcast_to(b, shape)[..., None, None], np.broadcast_to(a, shape)[..., None, None],", 0),
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
def test_matrix_pins_catch_mutant(mid, old, new, occ, tmp_path):
    src = open(SRC).read()
    mutated = _mutate(src, old, new, occ)
    assert mutated != src
    path = tmp_path / ("matrix_%s.py" % mid)
    path.write_text(mutated)
    spec = importlib.util.spec_from_file_location("matrix_mutant_%s" % mid, str(path))
    mutant = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mutant)
    caught = []
    for pin in matrix_pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError, FloatingPointError):   # noqa: PERF203
            caught.append(pin.__name__)
    assert caught, "no matrix pin caught the planted mistake %s" % mid
