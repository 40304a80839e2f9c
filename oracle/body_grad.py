"""CPU oracle for the gradient of an element scan with a body program --
TEST INFRASTRUCTURE (see ``oracle.body``; same import rules).

What it computes ("Nonlinear element scans", "Precision and gradients"):
gradients flow to `initial` and to every sequence; the gradient of a scan is
another element scan over the same lanes, run in the opposite trip order (a
reverse scan's from the first trip to the last), that applies the body's
vector-Jacobian product once a trip without forming the Jacobian;
comparisons and boolean casts have no derivative, `where` follows the
selected branch, the usual tie rules apply (a tie of `maximum` / `minimum`
splits the cotangent evenly, a tie of the reduction `max` among its equal
values); a width-one sequence (a parameter broadcast over the state) receives
the sum of its contributions.

Per trip, the body is evaluated again from the saved previous state onto a
tape (this module's own evaluator, which reproduces ``oracle.body`` bit for
bit), then swept backwards.  Readings (listed with the design notes):
  * every derivative is formed in f32 with the expressions below, each
    operation rounded: d(a+b) = (g, g); d(a-b) = (g, -g); d(a*b) = (g*b, g*a);
    d(a/b) = (g/b, -(g*q)/b) with q = a/b; d|a| = g * sign(a) (0 at 0);
    d sqrt = (g*0.5)/out; d exp = g*out; d log = g/a; d tanh = g*(1-out*out);
    d sin = g*cos(a); d cos = -(g*sin(a)); d rsqrt = g*((out*out*out)*-0.5);
    d acos = -(g/sqrt(1-a*a)); d asin = g/sqrt(1-a*a);
    d atan2(y, x) = ((g*x)/(x*x+y*y), -(g*y)/(x*x+y*y));
    d pow(a, b) = (g*(b*pow(a, b-1)), 0 if out == 0 else g*(out*log(a)));
    maximum / minimum: the larger (smaller) operand takes g, a tie or a NaN
    splits it as g*0.5 each; `where` passes g to the selected branch; `sum`
    passes g to every value; `max` passes g/count to each of its count equal
    maxima (none if the maximum is NaN);
  * contributions reach an operand in the tape's reverse order, each
    operand of a node in argument order, the first one assigned and later
    ones added; a width-one operand of a wide operation receives the sum of
    the wide contribution over w = 0..W-1 in order;
  * the state's cotangent entering a trip is (carried + output gradient).
"""
from __future__ import annotations

import math

import numpy as np

from .body import (Body, BodyError, Kw, Sym, Vec, _Ctx, _as_tensor, _ieee_maximum, _ieee_minimum, _is_num,
                   _keywords, _num_max, _NUMBER_BINARY, _NUMBER_COMPARE, _UNARY_F64, _NUMBER_UNARY, _COMPARE,
                   _via_f64)

__all__ = ["scan_body_backward"]

f32 = np.float32


class _T:
    """A tensor value on the tape: value [lanes, width] and how it was made."""

    __slots__ = ("v", "op", "args", "aux", "idx", "g")

    def __init__(self, v, op, args=(), aux=None):
        self.v = v
        self.op = op
        self.args = list(args)
        self.aux = aux
        self.idx = -1
        self.g = None


class _Tape:
    def __init__(self, ctx):
        self.ctx = ctx
        self.nodes = []

    def add(self, v, op, args=(), aux=None):
        t = _T(v, op, args, aux)
        t.idx = len(self.nodes)
        self.nodes.append(t)
        return t

    def const(self, v):
        """A plain number (or bool) meeting a tensor: a constant node."""
        return self.add(_as_tensor(v, self.ctx.lanes), "const")


def _fmul(a, b):
    return np.multiply(a, b, dtype=f32)


def _fadd(a, b):
    return np.add(a, b, dtype=f32)


def _fsub(a, b):
    return np.subtract(a, b, dtype=f32)


def _fdiv(a, b):
    with np.errstate(all="ignore"):
        return np.divide(a, b, dtype=f32)


def _sum_w(c):
    """Sum over the state's values in order w = 0..W-1 (a width-one result)."""
    acc = c[:, 0:1]
    for w in range(1, c.shape[1]):
        acc = _fadd(acc, c[:, w:w + 1])
    return acc


class _Evaluator:
    """The body's forward evaluation onto a tape.  It mirrors oracle.body's
    evaluator operation by operation (values must agree bit for bit)."""

    def __init__(self, tape):
        self.t = tape
        self.ctx = tape.ctx

    def tensor(self, v):
        return v if isinstance(v, _T) else self.t.const(v)

    def f32(self, v, what):
        t = self.tensor(v)
        if t.v.dtype != np.float32:
            raise BodyError("E-DIM-002", "%s wants f32, got bool" % what)
        return t

    def boolean(self, v, what):
        t = self.tensor(v)
        if t.v.dtype != np.bool_:
            raise BodyError("E-DIM-002", "%s wants bool, got f32" % what)
        return t

    def eval(self, form, env):
        ctx = self.ctx
        if isinstance(form, (bool, float)):
            return form
        if isinstance(form, Sym):
            if form not in env:
                raise BodyError("E-SCAN-001", "`%s` is not an argument of the body or a let binding" % form)
            return env[form]
        if isinstance(form, (Kw, Vec)) or not isinstance(form, list) or not form:
            raise BodyError("parse", "not a value")
        head, args = form[0], form[1:]
        if head == "let":
            inner = dict(env)
            for b in args[0]:
                inner[b[0]] = self.eval(b[1], inner)
            r = None
            for f in args[1:]:
                r = self.eval(f, inner)
            return r
        if head in ("sum", "max"):
            pos, kws = _keywords(args, (":axes", ":keepdims"))
            vals = [self.eval(p, env) for p in pos]
            if all(_is_num(v) for v in vals) and not kws:
                r = float(vals[0])
                for v in vals[1:]:
                    r = r + float(v) if head == "sum" else _num_max(r, float(v))
                return r
            a = self.f32(vals[0], head)
            axes = kws.get(":axes")
            if (axes is not None and len(axes) == 0) or a.v.shape[1] == 1:
                return a
            if head == "sum":
                return self.t.add(_sum_w(a.v), "sum", [a])
            acc = a.v[:, 0:1]
            for w in range(1, a.v.shape[1]):
                acc = _ieee_maximum(acc, a.v[:, w:w + 1])
            return self.t.add(acc, "rmax", [a])
        if head == "cast":
            v = self.tensor(self.eval(args[0], env))
            if args[1] == ":f32":
                return v if v.v.dtype == np.float32 else self.t.add(v.v.astype(f32), "nograd")
            return v if v.v.dtype == np.bool_ else self.t.add(v.v != f32(0), "nograd")
        if head in ("broadcast-to", "reshape"):
            v = self.eval(args[0], env)
            dims = args[1]
            if not isinstance(v, _T):
                return v
            if head == "broadcast-to" and len(dims) >= 1 and v.v.shape[1] == 1 and ctx.vector and dims[-1] == ctx.W:
                return self.t.add(np.repeat(v.v, ctx.W, axis=1), "bcast", [v])
            return v
        vals = [self.eval(a, env) for a in args]
        if head in ("+", "*", "-", "/"):
            if len(vals) == 1:
                v = vals[0]
                if _is_num(v):
                    return {"+": v, "*": v, "-": -v}.get(head) if head != "/" else _NUMBER_BINARY["/"](1.0, v)
                t = self.f32(v, head)
                if head == "-":
                    return self.t.add(np.negative(t.v), "neg", [t])
                if head == "/":
                    one = self.t.const(1.0)
                    return self.t.add(_fdiv(one.v, t.v), "div", [one, t])
                return t
            acc = vals[0]
            for v in vals[1:]:
                if _is_num(acc) and _is_num(v):
                    acc = _NUMBER_BINARY[head](acc, v)
                else:
                    a, b = self.f32(acc, head), self.f32(v, head)
                    fn = {"+": _fadd, "-": _fsub, "*": _fmul, "/": _fdiv}[head]
                    acc = self.t.add(fn(a.v, b.v), {"+": "add", "-": "sub", "*": "mul", "/": "div"}[head], [a, b])
            return acc
        if head in _COMPARE:
            a, b = vals
            if _is_num(a) and _is_num(b):
                return _NUMBER_COMPARE[head](a, b)
            a, b = self.f32(a, head), self.f32(b, head)
            return self.t.add(_COMPARE[head](a.v, b.v), "nograd")
        if head in ("and", "or"):
            ts = [self.boolean(v, head) for v in vals]
            acc = ts[0].v
            for t in ts[1:]:
                acc = (acc & t.v) if head == "and" else (acc | t.v)
            return self.t.add(acc, "nograd")
        if head == "not":
            return self.t.add(~self.boolean(vals[0], "not").v, "nograd")
        if head == "where":
            m = self.boolean(vals[0], "where")
            a, b = self.tensor(vals[1]), self.tensor(vals[2])
            return self.t.add(np.where(m.v, a.v, b.v), "where", [a, b], aux=m.v)
        if head in ("neg", "abs"):
            a = self.f32(vals[0], head)
            return self.t.add(np.negative(a.v) if head == "neg" else np.abs(a.v), head, [a])
        if head == "sqrt":
            if _is_num(vals[0]):
                x = vals[0]
                return math.sqrt(x) if x >= 0 else math.nan
            a = self.f32(vals[0], head)
            with np.errstate(all="ignore"):
                return self.t.add(np.sqrt(a.v), "sqrt", [a])
        if head in _UNARY_F64:
            if head in _NUMBER_UNARY and _is_num(vals[0]):
                with np.errstate(all="ignore"):
                    return float(_UNARY_F64[head](np.float64(vals[0])))
            a = self.f32(vals[0], head)
            return self.t.add(_via_f64(_UNARY_F64[head], a.v), head, [a])
        if head in ("pow", "atan2", "maximum", "minimum"):
            if head == "pow" and _is_num(vals[0]) and _is_num(vals[1]):
                with np.errstate(all="ignore"):
                    return float(np.power(np.float64(vals[0]), np.float64(vals[1])))
            a, b = self.f32(vals[0], head), self.f32(vals[1], head)
            if head == "pow":
                return self.t.add(_via_f64(np.power, a.v, b.v), "pow", [a, b])
            if head == "atan2":
                return self.t.add(_via_f64(np.arctan2, a.v, b.v), "atan2", [a, b])
            av, bv = np.broadcast_arrays(a.v, b.v)
            fn = _ieee_maximum if head == "maximum" else _ieee_minimum
            return self.t.add(fn(av, bv), head, [a, b])
        raise BodyError("op", "`%s` is not an operation a body may use" % head)


def _contributions(node):
    """(operand, contribution) pairs of a node with cotangent g, in operand order."""
    g = node.g
    op = node.op
    a = node.args[0] if node.args else None
    b = node.args[1] if len(node.args) > 1 else None
    out = node.v
    if op == "add":
        return [(a, g), (b, g)]
    if op == "sub":
        return [(a, g), (b, np.negative(g))]
    if op == "mul":
        return [(a, _fmul(g, b.v)), (b, _fmul(g, a.v))]
    if op == "div":
        return [(a, _fdiv(g, b.v)), (b, np.negative(_fdiv(_fmul(g, out), b.v)))]
    if op == "neg":
        return [(a, np.negative(g))]
    if op == "abs":
        zero = np.zeros_like(g)
        return [(a, np.where(a.v > 0, g, np.where(a.v < 0, np.negative(g), zero)))]
    if op == "sqrt":
        return [(a, _fdiv(_fmul(g, f32(0.5)), out))]
    if op == "exp":
        return [(a, _fmul(g, out))]
    if op == "log":
        return [(a, _fdiv(g, a.v))]
    if op == "tanh":
        return [(a, _fmul(g, _fsub(f32(1.0), _fmul(out, out))))]
    if op == "sin":
        return [(a, _fmul(g, _via_f64(np.cos, a.v)))]
    if op == "cos":
        return [(a, np.negative(_fmul(g, _via_f64(np.sin, a.v))))]
    if op == "rsqrt":
        return [(a, _fmul(g, _fmul(_fmul(_fmul(out, out), out), f32(-0.5))))]
    if op in ("acos", "asin"):
        with np.errstate(all="ignore"):
            s = np.sqrt(_fsub(f32(1.0), _fmul(a.v, a.v)))
        c = _fdiv(g, s)
        return [(a, np.negative(c) if op == "acos" else c)]
    if op == "atan2":
        den = _fadd(_fmul(b.v, b.v), _fmul(a.v, a.v))        # x*x + y*y (a = y, b = x)
        return [(a, _fdiv(_fmul(g, b.v), den)), (b, np.negative(_fdiv(_fmul(g, a.v), den)))]
    if op == "pow":
        pw = _via_f64(np.power, a.v, _fsub(b.v, f32(1.0)))
        da = _fmul(g, _fmul(b.v, pw))
        lg = _via_f64(np.log, a.v)
        db = np.where(out == 0, f32(0.0), _fmul(g, _fmul(out, lg))).astype(f32)
        return [(a, da), (b, db)]
    if op in ("maximum", "minimum"):
        av, bv = np.broadcast_arrays(a.v, b.v)
        half = _fmul(g, f32(0.5))
        zero = np.zeros_like(g)
        if op == "maximum":
            a_wins, b_wins = av > bv, bv > av
        else:
            a_wins, b_wins = av < bv, bv < av
        ga = np.where(a_wins, g, np.where(b_wins, zero, half))
        gb = np.where(b_wins, g, np.where(a_wins, zero, half))
        return [(a, ga), (b, gb)]
    if op == "where":
        zero = np.zeros_like(g)
        m = node.aux
        return [(a, np.where(m, g, zero)), (b, np.where(m, zero, g))]
    if op == "sum":
        return [(a, np.broadcast_to(g, a.v.shape).astype(f32))]
    if op == "rmax":
        eq = a.v == out
        count = _sum_w(eq.astype(f32))
        zero = np.zeros_like(a.v)
        return [(a, np.where(eq, _fdiv(np.broadcast_to(g, a.v.shape), count), zero))]
    if op == "bcast":
        return [(a, g)]
    return []   # leaves, constants, booleans


def _accumulate(grads, operand, c):
    if operand.op in ("const", "nograd") or operand.v.dtype != np.float32:
        return
    c = np.asarray(c, dtype=f32)
    if operand.v.shape[1] == 1 and c.shape[1] != 1:
        c = _sum_w(c)                     # a width-one operand of a wide operation
    if c.shape != operand.v.shape:
        c = np.ascontiguousarray(np.broadcast_to(c, operand.v.shape))
    prev = grads.get(operand.idx)
    grads[operand.idx] = c if prev is None else _fadd(prev, c)


def trip_vjp(body: Body, ctx: _Ctx, p, seq_vals, lam):
    """One trip's VJP: (cotangent of the previous state, [cotangent of each
    sequence's value]) for the body evaluated at state p."""
    tape = _Tape(ctx)
    h = tape.add(p, "state")
    seqs = [tape.add(v, "seq") for v in seq_vals]
    env = {body.params[0]: h}
    for name, s in zip(body.params[1:], seqs):
        env[name] = s
    ev = _Evaluator(tape)
    r = None
    for e in body.exprs:
        r = ev.eval(e, env)
    r = tape.const(r) if not isinstance(r, _T) else r
    grads = {}
    if r.op not in ("const", "nograd"):
        seed = lam if r.v.shape[1] == lam.shape[1] else _sum_w(lam)
        grads[r.idx] = np.asarray(seed, f32)
    for node in reversed(tape.nodes):
        if node.idx not in grads:
            continue
        node.g = grads[node.idx]
        for operand, c in _contributions(node):
            _accumulate(grads, operand, c)
    dp = grads.get(h.idx, np.zeros_like(p))
    ds = [grads.get(s.idx, np.zeros_like(s.v)) for s in seqs]
    return dp, ds, r.v


def scan_body_backward(text, initial, seqs, states, grad_out, axis=0, state_axis=False, reverse=False):
    """Gradients of sum(grad_out * scan) with respect to initial and every
    sequence, given the forward states.  Returns (grad_initial, [grad_seq])."""
    body = text if isinstance(text, Body) else Body(text)
    seqs = [np.ascontiguousarray(s, dtype=f32) for s in seqs]
    initial = np.asarray(initial, dtype=f32)
    states = np.asarray(states, dtype=f32)
    body.check(states.shape[-1] if state_axis else 1, [s.shape[-1] if state_axis else 1 for s in seqs],
               state_axis)
    grad_out = np.asarray(grad_out, dtype=f32)
    shape = list(states.shape)
    rank = len(shape)
    ax = axis + rank if axis < 0 else axis
    W = shape[-1] if state_axis else 1
    O = int(np.prod(shape[:ax], dtype=np.int64))
    T = shape[ax]
    J = int(np.prod(shape[ax + 1:], dtype=np.int64)) // W
    lanes = O * J
    widths = [s.shape[-1] if state_axis else 1 for s in seqs]
    sv = [s.reshape(O, T, J, w) for s, w in zip(seqs, widths)]
    hv = states.reshape(O, T, J, W)
    gv = grad_out.reshape(O, T, J, W)
    ctx = _Ctx(lanes, W, state_axis)
    g_seqs = [np.zeros((O, T, J, w), f32) for w in widths]
    lam = np.zeros((lanes, W), f32)
    # the backward scan runs opposite to the forward one
    order = range(T) if reverse else range(T - 1, -1, -1)
    for t in order:
        lam = _fadd(lam, gv[:, t].reshape(lanes, W))
        tp = t + 1 if reverse else t - 1
        p = initial.reshape(lanes, W) if (tp < 0 or tp >= T) else hv[:, tp].reshape(lanes, W)
        vals = [v[:, t].reshape(lanes, w) for v, w in zip(sv, widths)]
        dp, ds, _ = trip_vjp(body, ctx, p, vals, lam)
        for k, d in enumerate(ds):
            g_seqs[k][:, t] = d.reshape(O, J, widths[k])
        lam = np.asarray(dp, f32)
    return lam.reshape(initial.shape), [g.reshape(s.shape) for g, s in zip(g_seqs, seqs)]
