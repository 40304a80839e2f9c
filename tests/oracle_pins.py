"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each ``pin_*`` function takes a ``scan`` callable with the signature of
``oracle.scan`` and raises ``AssertionError`` when the oracle disagrees with
what the element-scan page ("Nonlinear element scans") and plain mathematics
fix.  ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutations.py`` runs them on deliberately broken builds of the
oracle and requires at least one pin to fail for each planted mistake.

The pins are independent restatements, not retypings of the oracle's loop:
  * hand-derived closed-form cases (``tests/golden/*.json``);
  * MAXPLUS by brute force: max over all suffixes (prefixes) of the
    sequentially rounded sums of costs, valid because f32 subtraction of a
    fixed number is monotone;
  * MAXPLUS with zero cost is a cumulative maximum (``np.maximum.accumulate``);
  * TANH_DECAY with zero decay is elementwise tanh; with small signals it is
    the first-order linear filter ``scipy.signal.lfilter``; with constant
    inputs it converges to the root of h = tanh(x + a h) (``brentq``);
  * NORMCAP with zero gate is x / max(1, ||x||) (``np.linalg.norm``); with
    small signals it is the same linear filter per component; every state
    has norm at most one;
  * structural identities from the page: reverse equals flip-scan-flip,
    chunked resume from a final-state slice, lane permutation, axis
    placement, and a width-one gate equals the gate materialised at width W.
"""
from __future__ import annotations

import glob
import json
import os

import numpy as np
import scipy.optimize
import scipy.signal

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
f32 = np.float32


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


# ---------------------------------------------------------------------------
# golden fixtures (hand-derived)

def golden_cases():
    """The element-scan fixtures (those naming a body; the directory also holds
    fixtures of other operations)."""
    out = []
    for p in sorted(glob.glob(os.path.join(GOLDEN, "*.json"))):
        with open(p) as f:
            c = json.load(f)
        if "body" in c:
            out.append(c)
    return out


def pin_golden(scan):
    cases = golden_cases()
    assert cases, "no golden fixtures found"
    for c in cases:
        got = scan(c["body"], np.array(c["initial"], f32),
                   [np.array(c["x"], f32), np.array(c["a"], f32)],
                   axis=c["axis"], state_axis=c["state_axis"], reverse=c["reverse"])
        want = np.array(c["expected"], np.float64)
        if c.get("bitwise"):
            assert_bitwise(got, want.astype(f32), c["name"])
        elif c["atol"] == 0.0:
            assert np.array_equal(got.astype(np.float64), want), (c["name"], got, want)
        else:
            err = np.max(np.abs(got.astype(np.float64) - want))
            assert err <= c["atol"], (c["name"], err, got, want)


# ---------------------------------------------------------------------------
# MAXPLUS

def _maxplus_brute_lane(x, c, init, reverse):
    """h[t] as a maximum over every starting point, by explicit f32 chains.

    Forward: candidates are x[s] for s <= t and the initial state, each
    lowered by c[s+1], ..., c[t] (the initial state by c[0], ..., c[t]) one
    rounded subtraction at a time.  Reverse mirrors this.
    """
    T = len(x)
    out = np.empty(T, f32)
    for t in range(T):
        cands = []
        if not reverse:
            starts = [(x[s], range(s + 1, t + 1)) for s in range(t + 1)]
            starts.append((init, range(0, t + 1)))
        else:
            starts = [(x[s], range(s - 1, t - 1, -1)) for s in range(t, T)]
            starts.append((init, range(T - 1, t - 1, -1)))
        for v0, steps in starts:
            v = f32(v0)
            for k in steps:
                v = f32(v - f32(c[k]))
            cands.append(v)
        best = cands[0]
        for v in cands[1:]:
            # IEEE maximum; +0 above -0 (inputs are NaN-free)
            if v > best or (v == best and np.signbit(best) and not np.signbit(v)):
                best = v
        out[t] = best
    return out


def pin_maxplus_bruteforce(scan):
    rng = _rng(11)
    # a small value set makes ties and signed zeros frequent
    vals = np.array([-1.0, -0.5, -0.25, -0.0, 0.0, 0.25, 0.5, 0.75, 1.0, 1e-8, 3.0], f32)
    costs = np.array([0.0, 0.0, 0.125, 0.25, 0.1, 1e-8, 0.5], f32)
    for trial in range(24):
        L = int(rng.integers(1, 5))
        T = int(rng.integers(1, 10))
        x = rng.choice(vals, size=(L, T)).astype(f32)
        c = rng.choice(costs, size=(L, T)).astype(f32)
        init = rng.choice(np.array([-3.0e38, -0.0, 0.0, 0.5, -2.0], f32), size=L).astype(f32)
        for reverse in (False, True):
            got = scan("MAXPLUS", init, [x, c], axis=1, reverse=reverse)
            want = np.stack([_maxplus_brute_lane(x[l], c[l], init[l], reverse) for l in range(L)])
            assert_bitwise(got, want, "maxplus brute force trial %d reverse=%s" % (trial, reverse))


def pin_maxplus_zero_cost_is_cummax(scan):
    rng = _rng(12)
    x = rng.uniform(-1, 1, size=(5, 33)).astype(f32)
    c = np.zeros_like(x)
    init = rng.uniform(-0.5, 0.5, size=5).astype(f32)
    fwd = scan("MAXPLUS", init, [x, c], axis=1)
    want = np.maximum.accumulate(np.concatenate([init[:, None], x], axis=1), axis=1)[:, 1:]
    assert_bitwise(fwd, want, "forward cummax")
    rev = scan("MAXPLUS", init, [x, c], axis=1, reverse=True)
    xr = np.concatenate([x, init[:, None]], axis=1)[:, ::-1]
    want = np.maximum.accumulate(xr, axis=1)[:, ::-1][:, :-1]
    assert_bitwise(rev, want, "reverse cummax")


# ---------------------------------------------------------------------------
# TANH_DECAY

def pin_tanh_zero_decay(scan):
    rng = _rng(21)
    x = rng.normal(0, 2, size=(4, 17)).astype(f32)
    a = np.zeros_like(x)
    init = rng.normal(0, 1, size=4).astype(f32)
    got = scan("TANH_DECAY", init, [x, a], axis=1)
    want = np.tanh(x.astype(np.float64)).astype(f32)
    assert_bitwise(got, want, "tanh with zero decay")


def pin_tanh_small_signal_filter(scan):
    """|x + a h| << 1: tanh(v) = v (1 + O(v^2)), so the scan is the IIR filter
    h[t] = x[t] + a h[t-1] (per lane constant a), forward and reverse."""
    rng = _rng(22)
    L, T = 6, 40
    a_lane = rng.uniform(-0.9, 0.9, size=L)
    x = (1e-4 * rng.normal(size=(L, T))).astype(f32)
    a = np.repeat(a_lane[:, None], T, axis=1).astype(f32)
    init = (1e-4 * rng.normal(size=L)).astype(f32)
    for reverse in (False, True):
        got = scan("TANH_DECAY", init, [x, a], axis=1, reverse=reverse).astype(np.float64)
        want = np.empty((L, T))
        for l in range(L):
            al = float(a[l, 0])
            xs = x[l, ::-1] if reverse else x[l]
            y, _ = scipy.signal.lfilter([1.0], [1.0, -al], xs.astype(np.float64),
                                        zi=[al * float(init[l])])
            want[l] = y[::-1] if reverse else y
        scale = np.max(np.abs(want))
        err = np.max(np.abs(got - want))
        assert err <= 1e-5 * scale, ("tanh small-signal filter", reverse, err, scale)


def pin_tanh_fixed_point(scan):
    """Constant x and |a| < 1: the step map contracts, so h converges to the
    unique root of h = tanh(x + a h)."""
    rng = _rng(23)
    L, T = 5, 400
    xs = rng.normal(0, 1, size=L)
    as_ = rng.uniform(-0.8, 0.8, size=L)
    x = np.repeat(xs[:, None], T, axis=1).astype(f32)
    a = np.repeat(as_[:, None], T, axis=1).astype(f32)
    init = rng.uniform(-1, 1, size=L).astype(f32)
    got = scan("TANH_DECAY", init, [x, a], axis=1)
    for l in range(L):
        xl, al = float(x[l, 0]), float(a[l, 0])
        root = scipy.optimize.brentq(lambda h: h - np.tanh(xl + al * h), -1.0, 1.0, xtol=1e-15)
        assert abs(float(got[l, -1]) - root) <= 2e-6, ("tanh fixed point", l, got[l, -1], root)


def pin_tanh_range(scan):
    rng = _rng(24)
    x = rng.normal(0, 3, size=(8, 50)).astype(f32)
    a = rng.uniform(0.5, 0.99, size=(8, 50)).astype(f32)
    init = rng.normal(0, 0.1, size=8).astype(f32)
    got = scan("TANH_DECAY", init, [x, a], axis=1)
    assert np.all(np.abs(got) <= 1.0), "a tanh state left [-1, 1]"


# ---------------------------------------------------------------------------
# NORMCAP

def pin_normcap_zero_gate(scan):
    rng = _rng(31)
    B, T, H, W = 2, 9, 3, 16
    x = rng.normal(0, 0.5, size=(B, T, H, W)).astype(f32)
    g = np.zeros((B, T, H, 1), f32)
    init = rng.normal(0, 1, size=(B, H, W)).astype(f32)
    got = scan("NORMCAP", init, [x, g], axis=1, state_axis=True).astype(np.float64)
    xd = x.astype(np.float64)
    n = np.linalg.norm(xd, axis=-1, keepdims=True)
    want = xd / np.maximum(1.0, n)
    err = np.max(np.abs(got - want))
    assert err <= 1e-6, ("normcap with zero gate", err)


def pin_normcap_small_signal_filter(scan):
    """Norms stay below one, so the cap never acts and every component follows
    h_w[t] = a[t] h_w[t-1] + x_w[t]; per lane constant gate."""
    rng = _rng(32)
    B, T, H, W = 2, 30, 3, 8
    gate = rng.uniform(0.0, 0.9, size=(B, H))
    x = (1e-3 * rng.normal(size=(B, T, H, W))).astype(f32)
    g = np.broadcast_to(gate[:, None, :, None], (B, T, H, 1)).astype(f32)
    init = (1e-3 * rng.normal(size=(B, H, W))).astype(f32)
    for reverse in (False, True):
        got = scan("NORMCAP", init, [x, g], axis=1, state_axis=True, reverse=reverse).astype(np.float64)
        want = np.empty((B, T, H, W))
        for b in range(B):
            for hh in range(H):
                al = float(g[b, 0, hh, 0])
                for w in range(W):
                    xs = x[b, :, hh, w].astype(np.float64)
                    if reverse:
                        xs = xs[::-1]
                    y, _ = scipy.signal.lfilter([1.0], [1.0, -al], xs, zi=[al * float(init[b, hh, w])])
                    want[b, :, hh, w] = y[::-1] if reverse else y
        assert np.max(np.linalg.norm(want, axis=-1)) < 0.5
        err = np.max(np.abs(got - want))
        assert err <= 1e-5 * np.max(np.abs(want)), ("normcap small-signal filter", reverse, err)


def pin_normcap_full_width_gate_filter(scan):
    """A gate of full width W multiplies each component by its own value:
    with small signals every component is its own linear filter."""
    rng = _rng(35)
    B, T, H, W = 1, 20, 2, 4
    gate = rng.uniform(-0.9, 0.9, size=(B, H, W))
    x = (1e-3 * rng.normal(size=(B, T, H, W))).astype(f32)
    g = np.ascontiguousarray(np.broadcast_to(gate[:, None], (B, T, H, W))).astype(f32)
    init = (1e-3 * rng.normal(size=(B, H, W))).astype(f32)
    got = scan("NORMCAP", init, [x, g], axis=1, state_axis=True).astype(np.float64)
    want = np.empty((B, T, H, W))
    for hh in range(H):
        for w in range(W):
            al = float(g[0, 0, hh, w])
            y, _ = scipy.signal.lfilter([1.0], [1.0, -al], x[0, :, hh, w].astype(np.float64),
                                        zi=[al * float(init[0, hh, w])])
            want[0, :, hh, w] = y
    err = np.max(np.abs(got - want))
    assert err <= 1e-5 * np.max(np.abs(want)), ("normcap full-width gate", err)


def pin_normcap_norm_cap(scan):
    rng = _rng(33)
    B, T, H, W = 2, 64, 4, 16
    x = rng.normal(0, 3.0, size=(B, T, H, W)).astype(f32)
    g = rng.uniform(0.8, 1.0, size=(B, T, H, 1)).astype(f32)
    init = np.zeros((B, H, W), f32)
    got = scan("NORMCAP", init, [x, g], axis=1, state_axis=True).astype(np.float64)
    n = np.linalg.norm(got, axis=-1)
    # inputs of norm ~12 keep the cap active every trip: norms are one
    assert np.all(n <= 1.0 + 1e-6) and np.all(n >= 1.0 - 1e-6), (n.min(), n.max())
    # and the state points along the uncapped update y = g h + x
    prev = np.concatenate([init[:, None].astype(np.float64), got[:, :-1]], axis=1)
    y = g.astype(np.float64) * prev + x.astype(np.float64)
    cos = np.sum(y * got, axis=-1) / np.linalg.norm(y, axis=-1)
    assert np.all(cos >= 1.0 - 1e-6), cos.min()


def pin_normcap_width_one_is_clip(scan):
    """A one-value state has norm |y|: the cap is a clip to [-1, 1]."""
    rng = _rng(34)
    B, T = 3, 25
    x = rng.normal(0, 1.0, size=(B, T, 1)).astype(f32)
    g = rng.uniform(0.5, 1.0, size=(B, T, 1)).astype(f32)
    init = rng.uniform(-1, 1, size=(B, 1)).astype(f32)
    got = scan("NORMCAP", init, [x, g], axis=1, state_axis=True)
    h = init[:, 0].copy()
    for t in range(T):
        h = np.clip(g[:, t, 0] * h + x[:, t, 0], f32(-1), f32(1)).astype(f32)
        assert_bitwise(got[:, t, 0], h, "normcap width one, trip %d" % t)


# ---------------------------------------------------------------------------
# structure shared by all bodies

def _case(body, rng, shape=(3, 13, 5, 4), axis=1, state_axis=False):
    if body == "NORMCAP":
        state_axis = True
    x = rng.normal(0, 1, size=shape).astype(f32)
    if body == "MAXPLUS":
        x = rng.uniform(-1, 1, size=shape).astype(f32)
        a = rng.uniform(0, 0.1, size=shape).astype(f32)
    elif body == "NORMCAP":
        a = rng.uniform(0.8, 1.0, size=shape[:-1] + (1,)).astype(f32)
    else:
        a = rng.uniform(0.5, 0.99, size=shape).astype(f32)
    ax = axis % len(shape)
    init = rng.normal(0, 0.3, size=shape[:ax] + shape[ax + 1:]).astype(f32)
    return init, x, a, state_axis


BODY_LIST = ("TANH_DECAY", "NORMCAP", "MAXPLUS")


def pin_reverse_is_flip_scan_flip(scan):
    rng = _rng(41)
    for body in BODY_LIST:
        init, x, a, sa = _case(body, rng)
        rev = scan(body, init, [x, a], axis=1, state_axis=sa, reverse=True)
        fwd = scan(body, init, [np.flip(x, 1), np.flip(a, 1)], axis=1, state_axis=sa)
        assert_bitwise(rev, np.flip(fwd, 1), body + " reverse vs flip-scan-flip")


def pin_final_state_and_chunked_resume(scan):
    """The state after the last trip sits at position T-1 (forward) or 0
    (reverse); feeding it as the next call's initial state continues the
    recurrence exactly."""
    rng = _rng(42)
    for body in BODY_LIST:
        init, x, a, sa = _case(body, rng)
        T = x.shape[1]
        t0 = 6
        full = scan(body, init, [x, a], axis=1, state_axis=sa)
        first = scan(body, init, [x[:, :t0], a[:, :t0]], axis=1, state_axis=sa)
        second = scan(body, first[:, t0 - 1], [x[:, t0:], a[:, t0:]], axis=1, state_axis=sa)
        assert_bitwise(np.concatenate([first, second], 1), full, body + " forward resume")
        rfull = scan(body, init, [x, a], axis=1, state_axis=sa, reverse=True)
        rlast = scan(body, init, [x[:, t0:], a[:, t0:]], axis=1, state_axis=sa, reverse=True)
        rfirst = scan(body, rlast[:, 0], [x[:, :t0], a[:, :t0]], axis=1, state_axis=sa, reverse=True)
        assert_bitwise(np.concatenate([rfirst, rlast], 1), rfull, body + " reverse resume")
        # one trip from initial equals the first output of the long scan
        one = scan(body, init, [x[:, :1], a[:, :1]], axis=1, state_axis=sa)
        assert_bitwise(one[:, 0], full[:, 0], body + " single trip")
        assert T > t0


def pin_lane_permutation(scan):
    rng = _rng(43)
    for body in BODY_LIST:
        init, x, a, sa = _case(body, rng)
        perm = rng.permutation(x.shape[0])
        base = scan(body, init, [x, a], axis=1, state_axis=sa)
        got = scan(body, init[perm], [x[perm], a[perm]], axis=1, state_axis=sa)
        assert_bitwise(got, base[perm], body + " lane permutation")
        # permuting the lanes after the axis (not the state axis)
        perm2 = rng.permutation(x.shape[2])
        got = scan(body, init[:, perm2], [x[:, :, perm2], a[:, :, perm2]], axis=1, state_axis=sa)
        assert_bitwise(got, base[:, :, perm2], body + " inner lane permutation")


def pin_axis_placement(scan):
    """The scan along axis k of a tensor equals the scan along axis 0 of the
    same tensor with axis k moved to the front (C-contiguous layouts differ)."""
    rng = _rng(44)
    for body in BODY_LIST:
        _, x, a, sa = _case(body, rng, shape=(3, 4, 11, 2))
        nd = x.ndim
        axes = list(range(nd - 1)) + [-nd, -2] if sa else list(range(-nd, nd))
        for ax in axes:
            axp = ax % nd
            init = rng.normal(0, 0.3, size=x.shape[:axp] + x.shape[axp + 1:]).astype(f32)
            got = scan(body, init, [x, a], axis=ax, state_axis=sa)
            xm = np.ascontiguousarray(np.moveaxis(x, axp, 0))
            am = np.ascontiguousarray(np.moveaxis(a, axp, 0))
            ref = scan(body, init, [xm, am], axis=0, state_axis=sa)
            assert_bitwise(got, np.moveaxis(ref, 0, axp), "%s axis %d" % (body, ax))


def pin_gate_broadcast(scan):
    """A width-one sequence under a state axis acts as the same value at every
    state position, i.e. equals the sequence repeated to width W."""
    rng = _rng(45)
    B, T, H, W = 2, 11, 3, 5
    for body in BODY_LIST:
        x = rng.normal(0, 1, size=(B, T, H, W)).astype(f32)
        g = rng.uniform(0.5, 1.0, size=(B, T, H, 1)).astype(f32)
        init = rng.normal(0, 0.3, size=(B, H, W)).astype(f32)
        narrow = scan(body, init, [x, g], axis=1, state_axis=True)
        wide = scan(body, init, [x, np.ascontiguousarray(np.repeat(g, W, axis=-1))], axis=1, state_axis=True)
        assert_bitwise(narrow, wide, body + " width-one gate")
        if body != "NORMCAP":
            # pointwise bodies: a vector state is W independent scalar lanes
            scalar = scan(body, init, [x, np.ascontiguousarray(np.repeat(g, W, axis=-1))], axis=1)
            assert_bitwise(narrow, scalar, body + " vector state vs scalar lanes")


def pin_f64_twin_close(scan):
    """Diagnostic: the f32 recurrence stays within the float tolerance of the
    same recurrence in f64."""
    _np = np
    rng = _rng(46)
    for body in BODY_LIST:
        init, x, a, sa = _case(body, rng, shape=(2, 200, 3, 16))
        r32 = scan(body, init, [x, a], axis=1, state_axis=sa).astype(_np.float64)
        r64 = scan(body, init, [x, a], axis=1, state_axis=sa, dtype=_np.float64)
        err = _np.max(_np.abs(r32 - r64) / (1.0 + _np.abs(r64)))
        assert err <= 1e-5, (body, err)




# ---------------------------------------------------------------------------
# backward pass ("Precision and gradients": gradients reach initial and every
# sequence; the gradient is a scan in the opposite direction)

def _fd_case(body, rng, W=None, gate_wide=False):
    """Small random case in f64-friendly ranges, with no MAXPLUS ties."""
    if body == "NORMCAP":
        W = W or 4
        shape = (2, 6, 3, W)
        x = rng.normal(0, 0.6, size=shape)
        g = rng.uniform(0.6, 1.0, size=shape if gate_wide else shape[:-1] + (1,))
        init = rng.normal(0, 0.3, size=(2, 3, W))
        return init, x, g, True
    shape = (2, 6, 3)
    if body == "MAXPLUS":
        x = rng.uniform(-1, 1, size=shape)
        c = rng.uniform(0.0, 0.3, size=shape)
        init = rng.uniform(-1, 1, size=(2, 3))
        return init, x, c, False
    x = rng.normal(0, 1, size=shape)
    a = rng.uniform(-0.9, 0.9, size=shape)
    init = rng.normal(0, 0.5, size=(2, 3))
    return init, x, a, False


def _fd_grads(scan, body, init, x, a, G, sa, reverse, eps=1e-6):
    """Central differences of L = sum(G * scan(...)) in the f64 twin."""
    def L(i_, x_, a_):
        return float(np.sum(G * scan(body, i_, [x_, a_], axis=1, state_axis=sa, reverse=reverse,
                                     dtype=np.float64)))
    out = []
    for which, arr in enumerate((init, x, a)):
        g = np.empty_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = [init.copy(), x.copy(), a.copy()]
            minus = [init.copy(), x.copy(), a.copy()]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            g[idx] = (L(*plus) - L(*minus)) / (2 * eps)
        out.append(g)
    return out


def pin_bwd_finite_differences(scan, scan_backward=None):
    """Every gradient matches central differences of the f64 forward."""
    if scan_backward is None:
        return
    rng = _rng(51)
    for body, kw in (("TANH_DECAY", {}), ("MAXPLUS", {}), ("NORMCAP", {}), ("NORMCAP", {"gate_wide": True})):
        for reverse in (False, True):
            init, x, a, sa = _fd_case(body, rng, **kw)
            init32, x32, a32 = init.astype(f32), x.astype(f32), a.astype(f32)
            init, x, a = init32.astype(np.float64), x32.astype(np.float64), a32.astype(np.float64)
            h = scan(body, init32, [x32, a32], axis=1, state_axis=sa, reverse=reverse)
            G = rng.normal(size=h.shape).astype(f32)
            gi, (gx, ga) = scan_backward(body, init32, [x32, a32], h, G, axis=1, state_axis=sa, reverse=reverse)
            fi, fx, fa = _fd_grads(scan, body, init, x, a, G.astype(np.float64), sa, reverse)
            for name, got, want in (("initial", gi, fi), ("x", gx, fx), ("a", ga, fa)):
                err = np.max(np.abs(got - want) / (1.0 + np.abs(want)))
                assert err <= 2e-4, (body, kw, reverse, name, err)


def pin_bwd_torch_autograd(scan, scan_backward=None):
    """Gradients equal autograd of a plain PyTorch loop of the same bodies
    (f64); MAXPLUS, whose gradient only routes and halves values, equals
    autograd in f32 exactly, ties included (maximum splits a tie evenly)."""
    if scan_backward is None:
        return
    import torch
    rng = _rng(52)

    def torch_scan(body, init, x, a, reverse):
        T = x.shape[1]
        h = init
        outs = [None] * T
        for s in range(T):
            t = T - 1 - s if reverse else s
            if body == "TANH_DECAY":
                h = torch.tanh(x[:, t] + a[:, t] * h)
            elif body == "MAXPLUS":
                h = torch.maximum(h - a[:, t], x[:, t])
            else:
                y = a[:, t] * h + x[:, t]
                n = torch.linalg.vector_norm(y, dim=-1, keepdim=True)
                h = y / torch.clamp(n, min=1.0)
            outs[t] = h
        return torch.stack(outs, 1)

    for body in BODY_LIST:
        for reverse in (False, True):
            init, x, a, sa = _fd_case(body, rng)
            init32, x32, a32 = init.astype(f32), x.astype(f32), a.astype(f32)
            h = scan(body, init32, [x32, a32], axis=1, state_axis=sa, reverse=reverse)
            G = rng.normal(size=h.shape).astype(f32)
            gi, (gx, ga) = scan_backward(body, init32, [x32, a32], h, G, axis=1, state_axis=sa, reverse=reverse)
            ts = [torch.tensor(v.astype(np.float64), requires_grad=True) for v in (init32, x32, a32)]
            out = torch_scan(body, *ts, reverse)
            want = torch.autograd.grad((out * torch.tensor(G.astype(np.float64))).sum(), ts)
            for name, got, w in zip(("initial", "x", "a"), (gi, gx, ga), want):
                w = w.numpy()
                err = np.max(np.abs(got - w) / (1.0 + np.abs(w)))
                assert err <= 1e-5, (body, reverse, name, err)
    # MAXPLUS with many ties, f32, exact
    vals = np.array([-1.0, -0.5, 0.0, 0.5, 1.0], f32)
    costs = np.array([0.0, 0.5], f32)
    for reverse in (False, True):
        x = rng.choice(vals, size=(3, 9, 4)).astype(f32)
        c = rng.choice(costs, size=(3, 9, 4)).astype(f32)
        init = rng.choice(vals, size=(3, 4)).astype(f32)
        h = scan("MAXPLUS", init, [x, c], axis=1, reverse=reverse)
        G = rng.choice(np.array([-2.0, 1.0, 0.25, 3.0], f32), size=h.shape).astype(f32)
        gi, (gx, gc) = scan_backward("MAXPLUS", init, [x, c], h, G, axis=1, reverse=reverse)
        ts = [torch.tensor(v, requires_grad=True) for v in (init, x, c)]
        out = torch_scan("MAXPLUS", *ts, reverse)
        want = torch.autograd.grad((out * torch.tensor(G)).sum(), ts)
        for name, got, w in zip(("initial", "x", "c"), (gi, gx, gc), want):
            assert np.array_equal(got, w.numpy()), ("maxplus ties", reverse, name)


def pin_bwd_tanh_zero_decay(scan, scan_backward=None):
    """With zero decay every trip is tanh of its own input: no cotangent
    reaches the initial state and dx = G (1 - h^2)."""
    if scan_backward is None:
        return
    rng = _rng(53)
    x = rng.normal(0, 1, size=(3, 8)).astype(f32)
    a = np.zeros_like(x)
    init = rng.normal(size=3).astype(f32)
    h = scan("TANH_DECAY", init, [x, a], axis=1)
    G = rng.normal(size=h.shape).astype(f32)
    gi, (gx, ga) = scan_backward("TANH_DECAY", init, [x, a], h, G, axis=1)
    assert np.all(gi == 0)
    t = np.tanh(x.astype(np.float64))
    assert np.max(np.abs(gx - G * (1 - t * t))) <= 1e-6


def pin_bwd_normcap_linear_adjoint(scan, scan_backward=None):
    """Inside the unit ball NORMCAP is the linear recurrence h = g h + x; its
    adjoint is the same first-order filter run backwards over the output
    gradient (scipy.signal.lfilter on the reversed sequence)."""
    if scan_backward is None:
        return
    rng = _rng(54)
    B, T, H, W = 2, 12, 3, 4
    gate = rng.uniform(0.2, 0.9, size=(B, H))
    x = (1e-3 * rng.normal(size=(B, T, H, W))).astype(f32)
    g = np.broadcast_to(gate[:, None, :, None], (B, T, H, 1)).astype(f32)
    init = (1e-3 * rng.normal(size=(B, H, W))).astype(f32)
    h = scan("NORMCAP", init, [x, g], axis=1, state_axis=True)
    G = rng.normal(size=h.shape).astype(f32)
    gi, (gx, gg) = scan_backward("NORMCAP", init, [x, g], h, G, axis=1, state_axis=True)
    for b in range(B):
        for hh in range(H):
            al = float(g[b, 0, hh, 0])
            for w in range(W):
                lam = scipy.signal.lfilter([1.0], [1.0, -al], G[b, ::-1, hh, w].astype(np.float64))[::-1]
                assert np.max(np.abs(gx[b, :, hh, w] - lam)) <= 1e-5 * (1 + np.max(np.abs(lam)))
                assert abs(gi[b, hh, w] - al * lam[0]) <= 1e-5 * (1 + abs(lam[0]))


BWD_PINS = [pin_bwd_finite_differences, pin_bwd_torch_autograd, pin_bwd_tanh_zero_decay,
            pin_bwd_normcap_linear_adjoint]
ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and not k.startswith("pin_bwd_")]
