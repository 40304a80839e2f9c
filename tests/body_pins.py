"""Pins of the body-program oracle (``oracle.body``) to facts from outside it.

Each ``pin_*`` takes ``scan_body`` (the signature of ``oracle.body.scan_body``)
and raises ``AssertionError`` when the result disagrees with what the pages
and plain mathematics fix.  ``test_body_oracle_pins.py`` runs them on the real
oracle; ``test_body_oracle_mutations.py`` plants mistakes in the oracle's
interpreter and requires a pin to catch each one.

The facts are independent of the interpreter:
  * the three bodies the element-scan page prints ("Nonlinear element
    scans": intro, `:state-axis` and `:reverse` examples) written as text give
    bit for bit what the fixed-body C oracle gives (itself pinned by its own
    closed forms, brute force and library routines);
  * bodies whose scans are library routines: running sums and products
    (``np.add.accumulate`` / ``np.multiply.accumulate``, sequential and so bit
    exact), running maxima, counts, ``np.logaddexp.accumulate``, the linear
    filter ``scipy.signal.lfilter``, angle wrapping, running Euclidean norms;
  * identities of the functions (rsqrt(x*x)*|x| = 1, acos(cos x) = x, ...);
  * hand-derived values for signed zeros, NaN and the folding of plain
    numbers at the front of `*` ("Tensor operations", overloaded
    arithmetic);
  * bodies that the "Arguments and body" contract rejects.
"""
from __future__ import annotations

import math

import numpy as np
import scipy.signal

f32 = np.float32

TANH_TEXT = "(lambda (h x a) (tanh (+ x (* a h))))"
MAXPLUS_TEXT = "(lambda (h x c) (maximum (- h c) x))"
NORMCAP_TEXT = """(lambda (h x a)
  (let ((y (+ (* a h) x)))
    (/ y (maximum 1.0 (sqrt (sum (* y y) :axes [-1]))))))"""


def _rng(seed):
    return np.random.default_rng(seed)


def _bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def assert_bitwise(got, want, what=""):
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = _bits(got) != _bits(want)
    assert not bad.any(), "%s: %d of %d values differ bitwise, first at %s: %r vs %r" % (
        what, int(bad.sum()), bad.size, np.argwhere(bad)[0], got[bad][0], want[bad][0])


def assert_close(got, want, tol, what=""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    err = np.abs(got - want) / (1.0 + np.abs(want))
    assert np.all(err <= tol), "%s: max scaled error %.3g > %.3g" % (what, float(err.max()), tol)


def _with_initial(init, seq):
    """[O, T, I] sequence with [O, I] initial prepended along the trips."""
    return np.concatenate([init[:, None, :], seq], axis=1)


# ---------------------------------------------------------------------------
# the pages' three bodies, as text, against the fixed-body C oracle

def pin_page_bodies_match_fixed_oracle(scan_body):
    import oracle
    rng = _rng(1)
    x = rng.standard_normal((3, 40, 9)).astype(f32)
    a = rng.uniform(0.5, 0.99, (3, 40, 9)).astype(f32)
    c = rng.uniform(0.0, 0.1, (3, 40, 9)).astype(f32)
    i0 = rng.standard_normal((3, 9)).astype(f32)
    for rev in (False, True):
        assert_bitwise(scan_body(TANH_TEXT, i0, [x, a], axis=1, reverse=rev),
                       oracle.scan(oracle.TANH_DECAY, i0, [x, a], axis=1, reverse=rev), "tanh text")
        assert_bitwise(scan_body(MAXPLUS_TEXT, i0, [x, c], axis=1, reverse=rev),
                       oracle.scan(oracle.MAXPLUS, i0, [x, c], axis=1, reverse=rev), "maxplus text")
    xv = (2 * rng.standard_normal((2, 30, 3, 8))).astype(f32)
    gv = rng.uniform(0.5, 1.0, (2, 30, 3, 1)).astype(f32)
    iv = (0.3 * rng.standard_normal((2, 3, 8))).astype(f32)
    for rev in (False, True):
        assert_bitwise(scan_body(NORMCAP_TEXT, iv, [xv, gv], axis=1, state_axis=True, reverse=rev),
                       oracle.scan(oracle.NORMCAP, iv, [xv, gv], axis=1, state_axis=True, reverse=rev),
                       "normcap text")


# ---------------------------------------------------------------------------
# bodies whose scans are library routines

def pin_running_sum_and_product(scan_body):
    rng = _rng(2)
    x = rng.standard_normal((2, 33, 5)).astype(f32)
    i0 = rng.standard_normal((2, 5)).astype(f32)
    want = np.add.accumulate(_with_initial(i0, x), axis=1, dtype=f32)[:, 1:]
    assert_bitwise(scan_body("(lambda (h x) (+ h x))", i0, [x], axis=1), want, "running sum")
    # reverse: the running sum from the end
    want_r = np.add.accumulate(_with_initial(i0, x[:, ::-1]), axis=1, dtype=f32)[:, 1:][:, ::-1]
    assert_bitwise(scan_body("(lambda (h x) (+ h x))", i0, [x], axis=1, reverse=True), want_r, "reverse sum")
    m = rng.uniform(0.8, 1.2, (2, 33, 5)).astype(f32)
    want = np.multiply.accumulate(_with_initial(i0, m), axis=1, dtype=f32)[:, 1:]
    assert_bitwise(scan_body("(lambda (h m) (* h m))", i0, [m], axis=1), want, "running product")


def pin_running_max_by_where(scan_body):
    rng = _rng(3)
    x = rng.permutation(np.arange(1, 4 * 50 + 1, dtype=np.float64)).reshape(4, 50).astype(f32)[..., None]
    i0 = np.full((4, 1), 10.5, f32)
    want = np.maximum.accumulate(_with_initial(i0, x), axis=1)[:, 1:]
    assert_bitwise(scan_body("(lambda (h x) (where (> x h) x h))", i0, [x], axis=1), want, "running max")
    # axis 0: a [T, lanes] layout
    xt = np.ascontiguousarray(x[..., 0].T)
    want0 = np.maximum.accumulate(np.concatenate([i0.T, xt], axis=0), axis=0)[1:]
    assert_bitwise(scan_body("(lambda (h x) (where (< h x) x h))", i0[:, 0], [xt], axis=0), want0, "axis 0")


def pin_counts_by_cast_and_logic(scan_body):
    rng = _rng(4)
    x = rng.uniform(0, 1, (3, 64, 4)).astype(f32)
    i0 = np.zeros((3, 4), f32)
    cnt = np.cumsum(x > f32(0.5), axis=1).astype(f32)
    assert_bitwise(scan_body("(lambda (h x) (+ h (cast (> x 0.5) :f32)))", i0, [x], axis=1), cnt, "count >")
    tails = np.cumsum((x > f32(0.9)) | (x < f32(0.1)), axis=1).astype(f32)
    assert_bitwise(scan_body("(lambda (h x) (where (or (> x 0.9) (< x 0.1)) (+ h 1) h))", i0, [x], axis=1),
                   tails, "count or")
    mid = np.cumsum((x >= f32(0.25)) & ~(x > f32(0.75)), axis=1).astype(f32)
    assert_bitwise(scan_body("(lambda (h x) (+ h (cast (and (>= x 0.25) (not (> x 0.75))) :f32)))", i0, [x],
                             axis=1), mid, "count and/not")
    ne = np.cumsum(np.round(x * 4) != 2, axis=1).astype(f32)
    xr = np.round(x * 4).astype(f32)
    assert_bitwise(scan_body("(lambda (h x) (+ h (cast (!= x 2) :f32)))", i0, [xr], axis=1), ne, "count !=")
    eq = np.cumsum(xr == 2, axis=1).astype(f32)
    assert_bitwise(scan_body("(lambda (h x) (+ h (cast (cast (= x 2) :f32) :f32)))", i0, [xr], axis=1), eq,
                   "count =")
    # each comparison on whole numbers, where ties occur
    for op, fn in (("<", np.less), ("<=", np.less_equal), (">", np.greater), (">=", np.greater_equal)):
        want = np.cumsum(fn(xr, 2), axis=1).astype(f32)
        assert_bitwise(scan_body("(lambda (h x) (+ (cast (%s x 2) :f32) h))" % op, i0, [xr], axis=1), want,
                       "count %s" % op)
    # f32 -> bool is "not zero", negative values included
    xc = (xr - 2).astype(f32)
    nz = np.cumsum(xc != 0, axis=1).astype(f32)
    assert_bitwise(scan_body("(lambda (h x) (+ h (cast (cast x :bool) :f32)))", i0, [xc], axis=1), nz,
                   "bool cast")


def pin_log_sum_exp(scan_body):
    rng = _rng(5)
    x = rng.standard_normal((2, 40, 3)).astype(f32)
    i0 = rng.standard_normal((2, 3)).astype(f32)
    want = np.logaddexp.accumulate(_with_initial(i0, x).astype(np.float64), axis=1)[:, 1:]
    got = scan_body("(lambda (h x) (log (+ (exp h) (exp x))))", i0, [x], axis=1)
    assert_close(got, want, 2e-6, "log-sum-exp")


def pin_linear_filter(scan_body):
    rng = _rng(6)
    x = rng.standard_normal((2, 200, 3)).astype(f32)
    i0 = rng.standard_normal((2, 3)).astype(f32)
    b0, a1 = float(f32(0.1)), float(f32(0.9))
    zi = np.broadcast_to((a1 * i0.astype(np.float64))[:, None, :], (2, 1, 3))
    want, _ = scipy.signal.lfilter([b0], [1.0, -a1], x.astype(np.float64), axis=1, zi=zi)
    got = scan_body("(lambda (h x) (+ (* 0.9 h) (* 0.1 x)))", i0, [x], axis=1)
    assert_close(got, want, 1e-5, "exponential average")
    # the same filter with the coefficients as sequences and a minus sign
    am = np.full_like(x, -0.9)
    got2 = scan_body("(lambda (h x m) (- (* 0.1 x) (* m h)))", i0, [x, am], axis=1)
    assert_close(got2, want, 1e-5, "filter with a sequence coefficient")


def pin_angle_wrap(scan_body):
    rng = _rng(7)
    x = rng.uniform(-1.0, 1.0, (3, 30, 4)).astype(f32)
    i0 = rng.uniform(-1.0, 1.0, (3, 4)).astype(f32)
    acc = i0.astype(np.float64)[:, None, :] + np.cumsum(x.astype(np.float64), axis=1)
    got = scan_body("(lambda (h x) (atan2 (sin (+ h x)) (cos (+ h x))))", i0, [x], axis=1).astype(np.float64)
    d = np.mod(got - acc + math.pi, 2 * math.pi) - math.pi
    assert np.all(np.abs(d) < 2e-5), float(np.abs(d).max())
    assert np.all(np.abs(got) <= math.pi + 1e-6)


def pin_running_norm(scan_body):
    rng = _rng(8)
    x = rng.standard_normal((2, 50, 3)).astype(f32)
    i0 = rng.standard_normal((2, 3)).astype(f32)
    want = np.sqrt(i0.astype(np.float64)[:, None, :] ** 2 + np.cumsum(x.astype(np.float64) ** 2, axis=1))
    assert_close(scan_body("(lambda (h x) (sqrt (+ (* h h) (* x x))))", i0, [x], axis=1), want, 1e-5, "sqrt")
    assert_close(scan_body("(lambda (h x) (pow (+ (pow h 2) (pow x 2.0)) 0.5))", i0, [x], axis=1), want, 1e-5,
                 "pow")


def pin_function_identities(scan_body):
    rng = _rng(9)
    x = rng.uniform(0.05, 3.0, (2, 20, 5)).astype(f32)
    s = np.where(rng.uniform(size=x.shape) < 0.5, -1, 1).astype(f32)
    i0 = np.zeros((2, 5), f32)
    one = scan_body("(lambda (h x) (* (rsqrt (* x x)) (abs x)))", i0, [x * s], axis=1)
    assert_close(one, np.ones_like(one), 1e-6, "rsqrt(x*x)*|x|")
    back = scan_body("(lambda (h x) (+ (* 0 h) (acos (cos x))))", i0, [x], axis=1)
    assert_close(back, x, 2e-6, "acos(cos x)")
    xs = (x - 1.5) / 1.6
    back = scan_body("(lambda (h x) (+ (asin (sin x)) (* h 0.0)))", i0, [xs.astype(f32)], axis=1)
    assert_close(back, xs, 2e-6, "asin(sin x)")
    th = scan_body("(lambda (h x) (- (tanh x) (neg h)))", i0, [xs.astype(f32)], axis=1)
    want = np.cumsum(np.tanh(xs.astype(np.float64)), axis=1)
    assert_close(th, want, 1e-5, "running sum of tanh")
    ex = scan_body("(lambda (h x) (/ (exp x) (/ h)))", np.ones_like(i0), [(x / 20).astype(f32)], axis=1)
    want = np.exp(np.cumsum((x / 20).astype(f32).astype(np.float64), axis=1))
    assert_close(ex, want, 1e-5, "exp products")


def pin_signed_zero_and_nan(scan_body):
    nan = float("nan")
    # maximum / minimum: +0 above -0, NaN propagates (IEEE 754-2019)
    xs = np.array([[[-0.0], [0.0], [-0.0], [1.0], [nan], [2.0]]], f32)   # [1, 6, 1]
    i0 = np.array([[0.0]], f32)
    mx = scan_body("(lambda (h x) (maximum h x))", i0, [xs], axis=1)
    want = np.array([[[0.0], [0.0], [0.0], [1.0], [nan], [nan]]], f32)
    assert_bitwise(np.nan_to_num(mx, nan=7.0), np.nan_to_num(want, nan=7.0), "maximum")
    assert not np.signbit(mx[0, 0, 0])
    # the same with -0 as the first operand
    mz = scan_body("(lambda (h x) (maximum h x))", np.array([[-0.0]], f32), [np.array([[[0.0]]], f32)], axis=1)
    assert not np.signbit(mz[0, 0, 0]), "maximum(-0, +0) is +0"
    mz = scan_body("(lambda (h x) (minimum h x))", np.array([[-0.0]], f32), [np.array([[[0.0]]], f32)], axis=1)
    assert np.signbit(mz[0, 0, 0]), "minimum(-0, +0) is -0"
    mn = scan_body("(lambda (h x) (minimum h x))", i0, [xs], axis=1)
    assert np.signbit(mn[0, 0, 0]) and mn[0, 0, 0] == 0, "minimum(+0, -0) is -0"
    assert np.isnan(mn[0, 4, 0]) and np.isnan(mn[0, 5, 0])
    # the comparisons are false on NaN, except !=
    z = np.zeros((1, 1), f32)
    for op, want_count in (("<", 0), ("<=", 0), (">", 0), (">=", 0), ("=", 0), ("!=", 1)):
        r = scan_body("(lambda (h x) (+ h (cast (%s x 0.0) :f32)))" % op, z, [np.array([[[nan]]], f32)], axis=1)
        assert r[0, 0, 0] == want_count, op
    # negation flips the sign of zero; abs clears it
    r = scan_body("(lambda (h x) (neg x))", z, [np.array([[[0.0]]], f32)], axis=1)
    assert np.signbit(r[0, 0, 0])
    r = scan_body("(lambda (h x) (abs x))", z, [np.array([[[-0.0]]], f32)], axis=1)
    assert not np.signbit(r[0, 0, 0])


def pin_number_folding(scan_body):
    """Plain numbers at the front of an n-ary `*` fold first ("Tensor
    operations", overloaded arithmetic): (* 3.0 0.1 x) multiplies x once by
    the f32 of the f64 product 0.30000000000000004, while (* x 3.0 0.1)
    rounds after each factor.  Numbers meet the tensor as f32 constants."""
    x = np.array([[[1.0], [3.0], [7.0], [0.1], [1e-3], [12345.678]]], f32)
    z = np.zeros((1, 1), f32)
    front = scan_body("(lambda (h x) (+ (* 0 h) (* 3.0 0.1 x)))", z, [x], axis=1)
    assert_bitwise(front, (f32(3.0 * 0.1) * x).astype(f32), "front numbers fold")
    back = scan_body("(lambda (h x) (+ (* 0 h) (* x 3.0 0.1)))", z, [x], axis=1)
    assert_bitwise(back, ((x * f32(3.0)).astype(f32) * f32(0.1)).astype(f32), "factors after a tensor")
    assert not np.array_equal(front, back), "the two orders must differ on these inputs"
    # numbers alone stay f64 until they meet the tensor: (+ 0.1 0.2) is the
    # f32 of 0.30000000000000004, (/ 1 3) the f32 of 1/3, (sqrt 2) f32(sqrt 2)
    r = scan_body("(lambda (h x) (+ (* 0 h) (* (+ 0.1 0.2) (/ 1 3) (sqrt 2) x)))", z, [x], axis=1)
    c = f32((0.1 + 0.2) * (1 / 3) * math.sqrt(2))
    assert_bitwise(r, (x * c).astype(f32), "number subexpressions")
    # 16777217 is not an f32: folded in f64 the product 50331651 rounds to
    # 50331652, while rounding each number first gives 16777216 * 3
    one = np.ones((1, 1, 1), f32)
    r = scan_body("(lambda (h x) (+ (* 0 h) (* 16777217 3 x)))", z, [one], axis=1)
    assert r[0, 0, 0] == f32(50331652.0), r[0, 0, 0]
    # an integer literal is the number; `-` with one argument negates
    r = scan_body("(lambda (h x) (- (* 2 x)))", z, [x], axis=1)
    assert_bitwise(r, -(f32(2) * x).astype(f32), "unary minus")
    r = scan_body("(lambda (h x) (/ x))", z, [x], axis=1)
    assert_bitwise(r, (f32(1) / x).astype(f32), "unary division")
    r = scan_body("(lambda (h x) (- x 1 2))", z, [x], axis=1)
    assert_bitwise(r, ((x - f32(1)).astype(f32) - f32(2)).astype(f32), "n-ary minus folds left")


def pin_let_in_order(scan_body):
    """`let` binds in order: (let ((y (+ h x)) (z (* y 2))) z) is h' = 2(h + x);
    with small integers every value is exact, so the closed form
    h_t = 2^t h_0 + sum_s 2^(t-s+1) x_s holds bit for bit."""
    rng = _rng(10)
    x = rng.integers(-4, 5, (3, 12, 2)).astype(f32)
    i0 = rng.integers(-3, 4, (3, 2)).astype(f32)
    got = scan_body("(lambda (h x) (let ((y (+ h x)) (z (* y 2))) z))", i0, [x], axis=1)
    xi = x.astype(np.int64)
    want = np.empty_like(xi)
    acc = i0.astype(np.int64)
    for t in range(12):
        acc = 2 * (acc + xi[:, t])
        want[:, t] = acc
    assert_bitwise(got, want.astype(f32), "let")
    # an inner binding shadows an argument
    got = scan_body("(lambda (h x) (let ((x (* x 0))) (+ h x)))", i0, [x], axis=1)
    assert_bitwise(got, np.broadcast_to(i0[:, None, :], x.shape), "shadowing")


def pin_vector_bodies(scan_body):
    """:state-axis bodies: reductions over the state and width-one gates."""
    rng = _rng(11)
    W = 6
    x = rng.standard_normal((2, 25, 3, W)).astype(f32)
    i0 = rng.standard_normal((2, 3, W)).astype(f32)
    # every component accumulates the sum of the trip's row
    want = i0.astype(np.float64)[:, None] + np.cumsum(x.astype(np.float64).sum(-1, keepdims=True), axis=1)
    got = scan_body("(lambda (h x) (+ h (sum x :axes [-1] :keepdims true)))", i0, [x], axis=1, state_axis=True)
    assert_close(got, want, 1e-5, "sum reduction")
    # the row maximum: exact
    rowmax = x.max(-1, keepdims=True)
    want = np.maximum.accumulate(np.concatenate([i0[:, None], np.broadcast_to(rowmax, x.shape)], axis=1),
                                 axis=1)[:, 1:]
    got = scan_body("(lambda (h x) (maximum h (max x :axes [0])))", i0, [x], axis=1, state_axis=True)
    assert_bitwise(got, want, "max reduction")
    # a width-one gate scales the whole state
    g = rng.uniform(0.9, 1.1, (2, 25, 3, 1)).astype(f32)
    want = np.multiply.accumulate(np.concatenate([i0[:, None], np.broadcast_to(g, x.shape)], axis=1),
                                  axis=1, dtype=f32)[:, 1:]
    assert_bitwise(scan_body("(lambda (h g) (* h g))", i0, [g], axis=1, state_axis=True), want, "gate")
    # the first values of a sum set its rounding: sequential order over w
    v = np.array([[[[1e8, 1.0, -1e8, 1.0]]]], f32)
    z = np.zeros((1, 1, 4), f32)
    got = scan_body("(lambda (h x) (+ (* h 0) (sum x)))", z, [v], axis=1, state_axis=True)
    assert_bitwise(got, np.full((1, 1, 1, 4), 1.0, f32), "sum order")
    # mean-centring: the state minus its mean has zero sum
    got = scan_body("(lambda (h x) (let ((y (+ h x))) (- y (/ (sum y) 6))))", i0, [x], axis=1,
                    state_axis=True)
    assert np.all(np.abs(got.astype(np.float64).sum(-1)) < 1e-5)
    # an explicit broadcast of a one-value vector to the state
    got = scan_body("(lambda (h x) (broadcast-to (sum (* h x) :keepdims true) [6]))", i0, [x], axis=1,
                    state_axis=True)
    assert np.all(got == got[..., :1])


def pin_reverse_is_flip(scan_body):
    rng = _rng(12)
    x = rng.standard_normal((2, 17, 3)).astype(f32)
    y = rng.standard_normal((2, 17, 3)).astype(f32)
    i0 = rng.standard_normal((2, 3)).astype(f32)
    body = "(lambda (h x y) (where (> (+ h x) y) (tanh (- h y)) (* 0.5 (+ h x))))"
    rev = scan_body(body, i0, [x, y], axis=1, reverse=True)
    fwd = scan_body(body, i0, [x[:, ::-1], y[:, ::-1]], axis=1)[:, ::-1]
    assert_bitwise(rev, fwd, "reverse = flip scan flip")


REJECTED = [
    # (state_axis, state width, sequence widths, text)
    (False, 1, [1], "(lambda (h x) (+ h y))"),                        # E-SCAN-001: unbound name
    (False, 1, [1], "(lambda (h x) (sum x))"),                        # a scalar state cannot reduce
    (False, 1, [1], "(lambda (h x) (tanh h x))"),                     # arity
    (False, 1, [1], "(lambda (h x) (> h x))"),                        # returns bool
    (False, 1, [1], "(lambda (h x) (where x h x))"),                  # mask is not bool
    (False, 1, [1], "(lambda (h x) (cast x :bf16))"),                 # casts only f32 <-> bool
    (False, 1, [1], "(lambda (h x) (matmul h x))"),                   # not a body operation
    (False, 1, [1], "(lambda (h x) (+ h (cast (> x 0) :f32))"),       # unbalanced
    (False, 1, [1], "(lambda (h) h)"),                                # no sequence
    (False, 1, [1], "(lambda (h x) (+ (> h x) 1))"),                  # arithmetic on bool
    (True, 4, [4], "(lambda (h x) (sum (* h x)))"),                   # returns width 1 for width 4
    (True, 4, [4], "(lambda (h x) (max h x))"),                       # max of two tensors
    (True, 4, [4], "(lambda (h x) (+ h (sum x :axes [0 -1])))"),      # an axis twice
    (True, 4, [4], "(lambda (h x) (+ h (sum x :axes [1])))"),         # no such axis
    (True, 4, [2], "(lambda (h x) (+ h x))"),                         # widths 4 and 2
]


def pin_rejected_bodies(scan_body):
    for state_axis, W, widths, text in REJECTED:
        i0 = np.zeros((1, W) if state_axis else (1,), f32)
        seqs = [np.zeros((1, 2, w) if state_axis else (1, 2), f32) for w in widths]
        try:
            scan_body(text, i0, seqs, axis=1, state_axis=state_axis)
        except Exception as e:   # the interpreter's BodyError (from whichever copy runs)
            if type(e).__name__ == "BodyError":
                continue
            raise
        raise AssertionError("accepted a body the contract rejects: %s" % text)


ALL_PINS = [
    pin_page_bodies_match_fixed_oracle,
    pin_running_sum_and_product,
    pin_running_max_by_where,
    pin_counts_by_cast_and_logic,
    pin_log_sum_exp,
    pin_linear_filter,
    pin_angle_wrap,
    pin_running_norm,
    pin_function_identities,
    pin_signed_zero_and_nan,
    pin_number_folding,
    pin_let_in_order,
    pin_vector_bodies,
    pin_reverse_is_flip,
    pin_rejected_bodies,
]
