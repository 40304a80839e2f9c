"""Pins of the body-program gradient oracle (``oracle.body_grad``).

  * the pages' three bodies written as text: the gradients of the fixed-body
    C oracle (itself pinned by finite differences, autograd and closed
    forms) -- TANH_DECAY and MAXPLUS bit for bit, NORMCAP (a different but
    equal formula) within 1e-6;
  * bodies written directly as PyTorch loops in f64, differentiated by
    autograd: gated tanh, log-sum-exp, running norms by sqrt and pow,
    rsqrt / abs / atan2 / sin / cos / minimum, and vector bodies with `sum`,
    `max` and width-one gates (whose gradient is summed over the state);
  * hand-derived ties: `maximum` splits evenly, the reduction `max` splits
    among its equal maxima;
  * the tape reproduces the forward scan bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

f32 = np.float32


def _rng(seed):
    return np.random.default_rng(seed)


def _scaled_err(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    return float(np.max(np.abs(got - want) / (1.0 + np.abs(want)))) if got.size else 0.0


def pin_page_bodies_match_fixed_oracle(scan_body, scan_body_backward):
    import oracle
    from body_pins import MAXPLUS_TEXT, NORMCAP_TEXT, TANH_TEXT
    rng = _rng(1)
    x = rng.standard_normal((3, 40, 9)).astype(f32)
    a = rng.uniform(0.5, 0.99, (3, 40, 9)).astype(f32)
    c = rng.uniform(0.0, 0.1, (3, 40, 9)).astype(f32)
    i0 = rng.standard_normal((3, 9)).astype(f32)
    G = rng.standard_normal((3, 40, 9)).astype(f32)
    for rev in (False, True):
        for text, body, seqs in ((TANH_TEXT, oracle.TANH_DECAY, [x, a]), (MAXPLUS_TEXT, oracle.MAXPLUS, [x, c])):
            st = scan_body(text, i0, seqs, axis=1, reverse=rev)
            gi, gs = scan_body_backward(text, i0, seqs, st, G, axis=1, reverse=rev)
            ci, cs = oracle.scan_backward(body, i0, seqs, st, G, axis=1, reverse=rev)
            assert np.array_equal(gi, ci) and all(np.array_equal(p, q) for p, q in zip(gs, cs)), (text, rev)
    xv = (2 * rng.standard_normal((2, 30, 3, 8))).astype(f32)
    gv = rng.uniform(0.5, 1.0, (2, 30, 3, 1)).astype(f32)
    iv = (0.3 * rng.standard_normal((2, 3, 8))).astype(f32)
    Gv = rng.standard_normal((2, 30, 3, 8)).astype(f32)
    for rev in (False, True):
        st = scan_body(NORMCAP_TEXT, iv, [xv, gv], axis=1, state_axis=True, reverse=rev)
        gi, gs = scan_body_backward(NORMCAP_TEXT, iv, [xv, gv], st, Gv, axis=1, state_axis=True, reverse=rev)
        ci, cs = oracle.scan_backward(oracle.NORMCAP, iv, [xv, gv], st, Gv, axis=1, state_axis=True, reverse=rev)
        assert _scaled_err(gi, ci) < 1e-6 and max(_scaled_err(p, q) for p, q in zip(gs, cs)) < 1e-6


# bodies as text and as PyTorch steps h' = f(h, *seq values) on [lanes, width] tensors
def _tmax(a, b):
    return torch.maximum(a, b)


AUTOGRAD_CASES = [
    # text, torch step, state width (0 scalar), sequence widths, ranges, initial range
    ("(lambda (h x a g) (where (> g 0.5) (tanh (+ x (* a h))) h))",
     lambda h, x, a, g: torch.where(g > 0.5, torch.tanh(x + a * h), h), 0, None,
     [(-1, 1), (0.5, 0.99), (0, 1)], (-1, 1)),
    ("(lambda (h x) (log (+ (exp h) (exp x))))", lambda h, x: torch.log(torch.exp(h) + torch.exp(x)), 0, None,
     [(-2, 2)], (-1, 1)),
    ("(lambda (h x) (sqrt (+ (* h h) (* x x))))", lambda h, x: torch.sqrt(h * h + x * x), 0, None,
     [(0.1, 1)], (0.5, 1)),
    ("(lambda (h x) (pow (+ (pow h 2) (pow x 2.0)) 0.5))", lambda h, x: (h ** 2 + x ** 2) ** 0.5, 0, None,
     [(0.1, 1)], (0.5, 1)),
    ("(lambda (h x) (- (* 0.5 h) (* (rsqrt (+ 1 (* x x))) (abs x))))",
     lambda h, x: 0.5 * h - torch.rsqrt(1 + x * x) * torch.abs(x), 0, None, [(-2, 2)], (-1, 1)),
    ("(lambda (h x) (atan2 (sin (+ h x)) (cos (* 0.5 (+ h x)))))",
     lambda h, x: torch.atan2(torch.sin(h + x), torch.cos(0.5 * (h + x))), 0, None, [(-0.1, 0.1)], (-0.5, 0.5)),
    ("(lambda (h x y) (minimum (+ h x) (- y h)))", lambda h, x, y: torch.minimum(h + x, y - h), 0, None,
     [(-1, 1), (-1, 1)], (-1, 1)),
    ("(lambda (h x) (/ (+ h x) (+ 2 (abs h))))", lambda h, x: (h + x) / (2 + torch.abs(h)), 0, None,
     [(-1, 1)], (-1, 1)),
    # vector states
    ("(lambda (h x g) (let ((y (+ (* g h) x))) (/ y (+ 1 (sqrt (sum (* y y)))))))",
     lambda h, x, g: (lambda y: y / (1 + torch.sqrt((y * y).sum(-1, keepdim=True))))(g * h + x), 4, [4, 1],
     [(-1, 1), (0.5, 1)], (-0.5, 0.5)),
    ("(lambda (h x) (let ((y (+ h x))) (- y (/ (sum y) 4))))",
     lambda h, x: (lambda y: y - y.sum(-1, keepdim=True) / 4)(h + x), 4, [4], [(-1, 1)], (-1, 1)),
    ("(lambda (h x g) (+ (* 0.5 h) (* g (max x :axes [-1] :keepdims true))))",
     lambda h, x, g: 0.5 * h + g * x.max(-1, keepdim=True).values, 8, [8, 1], [(-1, 1), (0.5, 1)], (-1, 1)),
    ("(lambda (h x) (tanh (+ h (* x (sum h :keepdims true)))))",
     lambda h, x: torch.tanh(h + x * h.sum(-1, keepdim=True)), 3, [3], [(-0.3, 0.3)], (-0.5, 0.5)),
]


def _draw(case, O, T, J, seed):
    _, _, W, widths, ranges, irange = case
    rng = _rng(seed)
    seqs = []
    for k, (lo, hi) in enumerate(ranges):
        shape = (O, T, J, widths[k]) if W else (O, T, J)
        seqs.append((lo + (hi - lo) * rng.random(shape)).astype(f32))
    lo, hi = irange
    initial = (lo + (hi - lo) * rng.random((O, J, W) if W else (O, J))).astype(f32)
    G = rng.standard_normal((O, T, J, W) if W else (O, T, J)).astype(f32)
    return initial, seqs, G


def pin_autograd_f64(scan_body, scan_body_backward):
    for ci, case in enumerate(AUTOGRAD_CASES):
        text, fn, W = case[0], case[1], case[2]
        for rev in (False, True):
            initial, seqs, G = _draw(case, 2, 12, 3, 100 + ci)
            st = scan_body(text, initial, seqs, axis=1, state_axis=W > 0, reverse=rev)
            gi, gs = scan_body_backward(text, initial, seqs, st, G, axis=1, state_axis=W > 0, reverse=rev)
            # the same recurrence written in torch, f64, differentiated by autograd
            ti = torch.tensor(initial, dtype=torch.float64, requires_grad=True)
            ts = [torch.tensor(s, dtype=torch.float64, requires_grad=True) for s in seqs]
            h = ti if W else ti
            outs = [None] * 12
            order = range(11, -1, -1) if rev else range(12)
            for t in order:
                h = fn(h, *[s[:, t] for s in ts])
                outs[t] = h
            loss = (torch.stack(outs, 1) * torch.tensor(G, dtype=torch.float64)).sum()
            loss.backward()
            assert _scaled_err(gi, ti.grad.numpy()) < 2e-4, (text, rev, _scaled_err(gi, ti.grad.numpy()))
            for k, (g, tsk) in enumerate(zip(gs, ts)):
                want = tsk.grad.numpy() if tsk.grad is not None else np.zeros(tsk.shape)   # only in a mask
                assert _scaled_err(g, want) < 2e-4, (text, rev, k, _scaled_err(g, want))


def pin_ties(scan_body, scan_body_backward):
    # maximum(h, x) with x equal to the incoming state: the cotangent splits evenly
    i0 = np.array([[0.5]], f32)
    x = np.array([[[0.5], [0.25], [2.0]]], f32)          # trip 0 ties (0.5 vs 0.5)
    st = scan_body("(lambda (h x) (maximum h x))", i0, [x], axis=1)
    G = np.array([[[1.0], [0.0], [0.0]]], f32)
    gi, (gx,) = scan_body_backward("(lambda (h x) (maximum h x))", i0, [x], st, G, axis=1)
    assert gi[0, 0] == 0.5 and gx[0, 0, 0] == 0.5 and gx[0, 1, 0] == 0.0, (gi, gx)
    # the reduction max: two equal maxima share the cotangent, the others get none
    v = np.array([[[[3.0, 1.0, 3.0, -2.0]]]], f32)
    z = np.zeros((1, 1, 4), f32)
    text = "(lambda (h x) (+ (* h 0) (max x :axes [0] :keepdims true)))"
    st = scan_body(text, z, [v], axis=1, state_axis=True)
    G = np.ones((1, 1, 1, 4), f32)
    _, (gx,) = scan_body_backward(text, z, [v], st, G, axis=1, state_axis=True)
    assert np.array_equal(gx[0, 0, 0], np.array([2.0, 0.0, 2.0, 0.0], f32)), gx
    # where follows the selected branch; the mask has no gradient
    text = "(lambda (h x) (where (> x 0) (* 2 x) (* 3 h)))"
    x = np.array([[[1.0], [-1.0], [1.0]]], f32)
    i0 = np.array([[1.0]], f32)
    st = scan_body(text, i0, [x], axis=1)
    G = np.ones((1, 3, 1), f32)
    gi, (gx,) = scan_body_backward(text, i0, [x], st, G, axis=1)
    # h1 = 2 x1, h2 = 3 h1, h3 = 2 x3 and L = h1 + h2 + h3: dL/dx1 = 2 + 3 * 2 = 8,
    # dL/dx2 = 0 (trip 2 takes h), dL/dx3 = 2; dL/dh0 = 0 (trip 1 takes x)
    assert np.array_equal(gx[0, :, 0], np.array([8.0, 0.0, 2.0], f32)) and gi[0, 0] == 0.0, (gx, gi)


def pin_tape_forward(scan_body, scan_body_backward):
    """The gradient oracle's own forward evaluation agrees with the forward
    oracle bit for bit (the tape differentiates what the scan computed)."""
    from oracle.body import Body, _Ctx
    from oracle.body_grad import trip_vjp
    for ci, case in enumerate(AUTOGRAD_CASES):
        text, W = case[0], case[2]
        initial, seqs, _ = _draw(case, 2, 5, 3, 200 + ci)
        st = scan_body(text, initial, seqs, axis=1, state_axis=W > 0)
        body = Body(text)
        Wd = W if W else 1
        ctx = _Ctx(6, Wd, W > 0)
        p = initial.reshape(6, Wd)
        for t in range(5):
            vals = [s[:, t].reshape(6, s.shape[-1] if W else 1) for s in seqs]
            _, _, out = trip_vjp(body, ctx, p, vals, np.zeros((6, Wd), f32))
            assert np.array_equal(np.broadcast_to(out, (6, Wd)), st[:, t].reshape(6, Wd)), (text, t)
            p = st[:, t].reshape(6, Wd)


ALL_PINS = [pin_page_bodies_match_fixed_oracle, pin_autograd_f64, pin_ties, pin_tape_forward]
