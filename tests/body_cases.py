"""Body programs used by the body-program tests, with seeded inputs.

Each case is a body text, its signature (scalar or vector state, the
sequences' widths) and the value range each sequence is drawn from.  ``exact``
marks bodies made only of IEEE-exact operations (+ - * / sqrt, comparisons,
where, casts, maximum/minimum, neg, abs): on the generic path (one thread per
lane, sums in state order) the GPU must then match the oracle bit for bit;
``exact_tiled`` adds that the lane-split skeletons keep that property (no
`sum` over a state split across threads).
"""
from __future__ import annotations

import numpy as np

f32 = np.float32

NORMCAP_TEXT = """(lambda (h x a)
  (let ((y (+ (* a h) x)))
    (/ y (maximum 1.0 (sqrt (sum (* y y) :axes [-1]))))))"""

# id, text, state width (0 = scalar state), sequence widths (None = full),
# ranges per sequence (lo, hi), initial range, exact, exact_tiled
CASES = [
    ("tanh_decay", "(lambda (h x a) (tanh (+ x (* a h))))", 0, None, [(-1, 1), (0.5, 0.99)], (-1, 1), False, False),
    ("maxplus", "(lambda (h x c) (maximum (- h c) x))", 0, None, [(-1, 1), (0, 0.1)], (-1, 1), True, True),
    ("average", "(lambda (h x) (+ (* 0.9 h) (* 0.1 x)))", 0, None, [(-2, 2)], (-1, 1), True, True),
    ("gated_tanh", "(lambda (h x a g) (where (> g 0.5) (tanh (+ x (* a h))) h))", 0, None,
     [(-1, 1), (0.5, 0.99), (0, 1)], (-1, 1), False, False),
    ("count_logic", "(lambda (h x) (+ h (cast (and (>= x 0.25) (not (> x 0.75))) :f32)))", 0, None, [(0, 1)],
     (0, 0), True, True),
    ("log_sum_exp", "(lambda (h x) (log (+ (exp h) (exp x))))", 0, None, [(-2, 2)], (-1, 1), False, False),
    ("angle", "(lambda (h x) (atan2 (sin (+ h x)) (cos (+ h x))))", 0, None, [(-0.01, 0.01)], (-1, 1), False,
     False),
    ("running_norm", "(lambda (h x) (sqrt (+ (* h h) (* x x))))", 0, None, [(-1, 1)], (0, 1), True, True),
    ("running_norm_pow", "(lambda (h x) (pow (+ (pow h 2) (pow x 2.0)) 0.5))", 0, None, [(-1, 1)], (0, 1), False,
     False),
    ("identities", "(lambda (h x) (+ (* 0.5 h) (* (rsqrt (* x x)) (abs x)) (acos (cos x)) (asin (* 0.5 x))))", 0,
     None, [(0.1, 2)], (0, 1), False, False),
    ("exp_product", "(lambda (h x) (* h (exp x)))", 0, None, [(-0.05, 0.05)], (0.5, 1.5), False, False),
    ("five_seqs", "(lambda (h a b c d e) (+ (* a h) (- b c) (* d e)))", 0, None,
     [(0.5, 0.9), (-1, 1), (-1, 1), (-1, 1), (-1, 1)], (-1, 1), True, True),
    ("eight_seqs", "(lambda (h a b c d e f g k) (minimum (+ (* a h) b c d) (maximum e (- f (* g k)))))", 0, None,
     [(0.5, 0.9)] + [(-1, 1)] * 7, (-1, 1), True, True),
    ("numbers_fold", "(lambda (h x) (+ (* 0.5 h) (* 3.0 0.1 x) (/ 1 3) (sqrt 2) (- 2)))", 0, None, [(-1, 1)],
     (-1, 1), True, True),
    # vector states
    ("normcap_w16", NORMCAP_TEXT, 16, [16, 1], [(-2, 2), (0.5, 1.0)], (-0.3, 0.3), True, False),
    ("normcap_w4_wide_gate", NORMCAP_TEXT, 4, [4, 4], [(-2, 2), (0.5, 1.0)], (-0.3, 0.3), True, False),
    ("row_max_w8", "(lambda (h x) (maximum h (max x :axes [0])))", 8, [8], [(-1, 1)], (-1, 1), True, True),
    ("gate_w8", "(lambda (h g) (* h g))", 8, [1], [(0.95, 1.05)], (-1, 1), True, True),
    ("centre_w4", "(lambda (h x) (let ((y (+ h x))) (- y (/ (sum y) 4))))", 4, [4], [(-1, 1)], (-1, 1), True,
     False),
    ("softsign_w2", "(lambda (h x g) (let ((y (+ (* g h) x))) (/ y (+ 1 (abs y)))))", 2, [2, 1],
     [(-1, 1), (0.5, 1)], (-1, 1), True, True),
    ("odd_width_w3", "(lambda (h x) (let ((y (+ h x))) (/ y (maximum 1.0 (sqrt (sum (* y y)))))))", 3, [3],
     [(-1, 1)], (-1, 1), True, True),
    ("width_one_state", "(lambda (h x) (+ (* 0.5 h) (sum x :keepdims true)))", 1, [1], [(-1, 1)], (-1, 1), True,
     True),
]

CASE_IDS = [c[0] for c in CASES]


def case(cid):
    for c in CASES:
        if c[0] == cid:
            return c
    raise KeyError(cid)


def make_inputs(c, O, T, J, seed=0, axis=1):
    """Seeded host inputs for a case: (initial, seqs, state_axis).

    Without a state axis the sequence shape is [O, T, J] (axis 1) or
    [O, J, T] (axis 2, the sequence axis last); with one it is [O, T, J, W]
    with each sequence's own last width."""
    _, _, W, widths, ranges, init_rng, _, _ = c
    rng = np.random.default_rng(seed)
    state_axis = W > 0
    seqs = []
    for k, (lo, hi) in enumerate(ranges):
        if state_axis:
            shape = (O, T, J, widths[k])
        else:
            shape = (O, T, J) if axis == 1 else (O, J, T)
        seqs.append((lo + (hi - lo) * rng.random(shape)).astype(f32))
    lo, hi = init_rng
    ishape = (O, J, W) if state_axis else (O, J)
    initial = (lo + (hi - lo) * rng.random(ishape)).astype(f32)
    return initial, seqs, state_axis
