"""CPU oracle for `element-scan` with a general body -- TEST INFRASTRUCTURE.

Like the rest of this package, only the test suite, ``__graft_entry__.smoke()``
and the bench's CPU-baseline and reference arms may import it.  It shares no
code with the CUDA library: the body text is read, checked and evaluated here
by its own small interpreter, vectorised over lanes with numpy and looping over
the trips in order.

What a body may contain follows "Nonlinear element scans", "Arguments and
body": pointwise arithmetic, transcendental functions, comparisons, `where`,
scalar constants, boolean intermediates and casts between f32 and bool; with
`:state-axis` the values are scalars or vectors of 1..16 values, `sum` and
`max` reduce a vector, and a one-value vector broadcasts against the state.
The operations and their names come from "Tensor operations", "Operations"
and "Shapes, dtypes, broadcasting" (the overloaded arithmetic, the six
comparisons, plain numbers at the front of an n-ary `*` folding first).

Readings where the pages leave a step open (each is also listed with the
design notes):
  * every tensor operation computes in f32 ("Precision and gradients") and
    rounds once: + - * / and sqrt are IEEE f32 operations; exp, log, tanh,
    sin, cos, acos, asin, atan2, pow and rsqrt are the f32 rounding of the
    function evaluated in f64 on the f32 operands;
  * plain numbers stay f64 host numbers while an overloaded operation sees
    only numbers (that is how numbers at the front of `*` fold first) and
    become f32 constants where they meet a tensor;
  * `maximum` / `minimum` are IEEE 754-2019 (+0 above -0, NaN propagates),
    the reduction `max` folds `maximum` over w = 0..W-1 and `sum` adds
    w = 0..W-1 in order, starting from the first value;
  * `max` with one argument (plus keywords) is the reduction; with two or
    more plain numbers it is their maximum; the elementwise pair is
    `maximum`;
  * the six comparisons are < <= > >= = !=; `and`, `or` and `not` combine
    booleans; (cast x :bool) is x != 0 and (cast b :f32) is 1 or 0;
  * `let` binds in order, each binding seeing the ones before it;
  * a name that is neither a lambda argument nor a `let` binding is E-SCAN-001
    (a parameter or context value read implicitly);
  * `(broadcast-to v shape)` and `(reshape v shape)` of a scalar are
    identities on the value; a broadcast whose last dimension is the state
    width makes a one-value vector a full-width one;
  * the body must return an f32 value as wide as the state.
"""
from __future__ import annotations

import math
import re

import numpy as np

__all__ = ["BodyError", "Body", "parse_body", "scan_body", "KNOWN_OPS"]


class BodyError(ValueError):
    """A body that the pages' contract rejects; ``code`` classifies it."""

    def __init__(self, code: str, msg: str):
        super().__init__("%s: %s" % (code, msg))
        self.code = code


# ---------------------------------------------------------------------------
# reader: s-expressions with numbers, symbols, keywords and [vectors]

_TOKEN = re.compile(r"\s*(?:(;[^\n]*)|([()\[\]])|([^\s()\[\];]+))")
_NUMBER = re.compile(r"^[+-]?(?:\d+\.?\d*|\.\d+)(?:[eE][+-]?\d+)?$")


class Sym(str):
    pass


class Kw(str):
    pass


class Vec(list):
    pass


def _tokens(text: str):
    pos = 0
    out = []
    while pos < len(text):
        m = _TOKEN.match(text, pos)
        if m is None or m.end() == pos:
            if text[pos:].strip() == "":
                break
            raise BodyError("parse", "unreadable text at %r" % text[pos:pos + 20])
        pos = m.end()
        if m.group(1) is not None:
            continue
        out.append(m.group(2) or m.group(3))
    return out


def _read(tokens, i):
    if i >= len(tokens):
        raise BodyError("parse", "unexpected end of body text")
    t = tokens[i]
    if t in "([":
        close = ")" if t == "(" else "]"
        items = []
        i += 1
        while True:
            if i >= len(tokens):
                raise BodyError("parse", "missing %r" % close)
            if tokens[i] == close:
                return (items if close == ")" else Vec(items)), i + 1
            if tokens[i] in ")]":
                raise BodyError("parse", "mismatched %r" % tokens[i])
            item, i = _read(tokens, i)
            items.append(item)
    if t in ")]":
        raise BodyError("parse", "unexpected %r" % t)
    if _NUMBER.match(t):
        return float(t), i + 1
    if t in ("true", "false"):
        return t == "true", i + 1
    if t.startswith(":"):
        return Kw(t), i + 1
    return Sym(t), i + 1


def read_sexpr(text: str):
    toks = _tokens(text)
    form, i = _read(toks, 0)
    if i != len(toks):
        raise BodyError("parse", "text after the body")
    return form


# ---------------------------------------------------------------------------
# values: a plain number (f64 float or bool) or a tensor over the lanes
# (np.float32 or np.bool_ array of shape [lanes, width], width 1 or W)

def _is_num(v):
    """A plain f64 number (a plain boolean is not one)."""
    return isinstance(v, float)


def _as_tensor(v, lanes):
    """A plain number meeting a tensor: an f32 (or bool) constant."""
    if isinstance(v, bool):
        return np.full((lanes, 1), v, dtype=np.bool_)
    if isinstance(v, float):
        return np.full((lanes, 1), np.float32(v), dtype=np.float32)
    return v


def _f32(v, lanes, what):
    t = _as_tensor(v, lanes)
    if t.dtype != np.float32:
        raise BodyError("E-DIM-002", "%s wants f32, got bool" % what)
    return t


def _bool(v, lanes, what):
    t = _as_tensor(v, lanes)
    if t.dtype != np.bool_:
        raise BodyError("E-DIM-002", "%s wants bool, got f32" % what)
    return t


def _widths_fit(ts, what):
    ws = {t.shape[1] for t in ts}
    if len(ws - {1}) > 1:
        raise BodyError("E-DIM-001", "%s: widths %s do not broadcast" % (what, sorted(ws)))


def _via_f64(fn, *ts):
    """f32 rounding of `fn` evaluated in f64 on f32 operands."""
    with np.errstate(all="ignore"):
        return fn(*[t.astype(np.float64) for t in ts]).astype(np.float32)


def _ieee_maximum(a, b):
    nan = np.isnan(a) | np.isnan(b)
    # equal values: only the zeros differ (+0 above -0)
    eq = np.where(np.signbit(a), b, a)
    r = np.where(a > b, a, np.where(b > a, b, eq))
    return np.where(nan, np.float32(np.nan), r).astype(np.float32)


def _ieee_minimum(a, b):
    nan = np.isnan(a) | np.isnan(b)
    eq = np.where(np.signbit(a), a, b)
    r = np.where(a < b, a, np.where(b < a, b, eq))
    return np.where(nan, np.float32(np.nan), r).astype(np.float32)


def _num_max(a, b):
    return a if a >= b or math.isnan(a) else b


# f32 elementwise operations (each rounds once)
def _add(a, b):
    return np.add(a, b, dtype=np.float32)


def _sub(a, b):
    return np.subtract(a, b, dtype=np.float32)


def _mul(a, b):
    return np.multiply(a, b, dtype=np.float32)


def _div(a, b):
    with np.errstate(all="ignore"):
        return np.divide(a, b, dtype=np.float32)


_TENSOR_BINARY = {"+": _add, "-": _sub, "*": _mul, "/": _div}
_NUMBER_BINARY = {
    "+": lambda a, b: a + b,
    "-": lambda a, b: a - b,
    "*": lambda a, b: a * b,
    "/": lambda a, b: float(np.divide(np.float64(a), np.float64(b))),
}

# tensor-only unaries and the overloaded ones, in f64 then rounded
_UNARY_F64 = {
    "exp": np.exp,
    "log": np.log,
    "tanh": np.tanh,
    "sin": np.sin,
    "cos": np.cos,
    "acos": np.arccos,
    "asin": np.arcsin,
    "rsqrt": lambda v: 1.0 / np.sqrt(v),
}
_NUMBER_UNARY = {"sqrt", "exp", "log"}     # overloaded: plain numbers stay numbers
_COMPARE = {
    "<": np.less, "<=": np.less_equal, ">": np.greater, ">=": np.greater_equal,
    "=": np.equal, "!=": np.not_equal,
}
_NUMBER_COMPARE = {
    "<": lambda a, b: a < b, "<=": lambda a, b: a <= b, ">": lambda a, b: a > b,
    ">=": lambda a, b: a >= b, "=": lambda a, b: a == b, "!=": lambda a, b: a != b,
}

KNOWN_OPS = sorted(
    ["+", "-", "*", "/", "pow", "sqrt", "exp", "log", "max", "sum", "neg", "rsqrt", "sin", "cos", "tanh", "abs",
     "acos", "asin", "atan2", "maximum", "minimum", "where", "cast", "and", "or", "not", "let", "broadcast-to",
     "reshape"] + list(_COMPARE))


class _Ctx:
    def __init__(self, lanes: int, state_width: int, vector_state: bool):
        self.lanes = lanes
        self.W = state_width
        self.vector = vector_state


def _keywords(args, allowed):
    pos, kws = [], {}
    i = 0
    while i < len(args):
        a = args[i]
        if isinstance(a, Kw):
            if a not in allowed:
                raise BodyError("arity", "unknown keyword %s" % a)
            if i + 1 >= len(args):
                raise BodyError("arity", "keyword %s has no value" % a)
            kws[a] = args[i + 1]
            i += 2
        else:
            pos.append(a)
            i += 1
    return pos, kws


def _reduce(op, pos, kws, vals, ctx):
    """(sum v) / (max v) of one tensor value: over the state's values."""
    if len(pos) != 1:
        if op == "max":
            raise BodyError("arity", "(max ...) over tensors takes one value; the elementwise pair is maximum")
        raise BodyError("arity", "(sum ...) over tensors takes one value")
    if not ctx.vector:
        raise BodyError("reduce", "a scalar state's body cannot reduce")
    axes = kws.get(":axes")
    if axes is not None:
        if not isinstance(axes, Vec) or not all(_is_num(a) and a == int(a) for a in axes):
            raise BodyError("E-DIM-001", ":axes takes a vector of integers")
        norm = [int(a) + 1 if a < 0 else int(a) for a in axes]
        if any(n != 0 for n in norm):
            raise BodyError("E-DIM-001", "a body value has one axis; :axes %s" % list(axes))
        if len(norm) != len(set(norm)):
            raise BodyError("E-DIM-001", "an axis is listed twice in :axes %s" % list(axes))
    keep = kws.get(":keepdims", False)
    if not isinstance(keep, bool):
        raise BodyError("arity", ":keepdims takes true or false")
    t = _f32(vals[0], ctx.lanes, "(%s ...)" % op)
    if axes is not None and len(axes) == 0:
        return t
    acc = t[:, 0:1]
    for w in range(1, t.shape[1]):
        acc = _add(acc, t[:, w:w + 1]) if op == "sum" else _ieee_maximum(acc, t[:, w:w + 1])
    return acc


def _eval(form, env, ctx):
    if isinstance(form, (bool, float)):
        return form
    if isinstance(form, Sym):
        if form not in env:
            raise BodyError("E-SCAN-001", "`%s` is not an argument of the body or a let binding" % form)
        return env[form]
    if isinstance(form, (Kw, Vec)):
        raise BodyError("parse", "%r is not a value" % (form,))
    if not isinstance(form, list) or len(form) == 0:
        raise BodyError("parse", "empty form")
    head, args = form[0], form[1:]
    if not isinstance(head, Sym):
        raise BodyError("parse", "a form starts with an operation name")
    L = ctx.lanes

    if head == "let":
        if len(args) < 2 or not isinstance(args[0], list):
            raise BodyError("arity", "(let ((name value) ...) body)")
        inner = dict(env)
        for b in args[0]:
            if not (isinstance(b, list) and len(b) == 2 and isinstance(b[0], Sym)):
                raise BodyError("arity", "a let binding is (name value)")
            inner[b[0]] = _eval(b[1], inner, ctx)
        r = None
        for f in args[1:]:
            r = _eval(f, inner, ctx)
        return r

    if head in ("sum", "max"):
        pos, kws = _keywords(args, (":axes", ":keepdims"))
        if len(pos) == 0:
            raise BodyError("arity", "(%s) needs a value" % head)
        vals = [_eval(p, env, ctx) for p in pos]
        if all(_is_num(v) for v in vals) and not kws:
            # plain numbers: their sum ("(sum xs) over a list of numbers adds
            # them") or their maximum
            r = float(vals[0])
            for v in vals[1:]:
                r = r + float(v) if head == "sum" else _num_max(r, float(v))
            return r
        return _reduce(head, pos, kws, vals, ctx)

    if head == "cast":
        if len(args) != 2 or not isinstance(args[1], Kw):
            raise BodyError("arity", "(cast x :f32) or (cast x :bool)")
        v = _as_tensor(_eval(args[0], env, ctx), L)
        if args[1] == ":f32":
            return v if v.dtype == np.float32 else v.astype(np.float32)
        if args[1] == ":bool":
            return v if v.dtype == np.bool_ else (v != np.float32(0))
        raise BodyError("E-DIM-002", "the body casts only between f32 and bool, not to %s" % args[1])
    if head in ("broadcast-to", "reshape"):
        if len(args) != 2 or not isinstance(args[1], Vec) or not all(_is_num(d) for d in args[1]):
            raise BodyError("arity", "(%s value [dims...])" % head)
        v = _eval(args[0], env, ctx)
        dims = args[1]
        if _is_num(v) or isinstance(v, bool):
            return v
        if head == "broadcast-to" and len(dims) >= 1 and v.shape[1] == 1 and ctx.vector and dims[-1] == ctx.W:
            return np.repeat(v, ctx.W, axis=1)
        return v

    vals = [_eval(a, env, ctx) for a in args]

    def arity(n_lo, n_hi=None):
        n_hi = n_lo if n_hi is None else n_hi
        if len(vals) < n_lo or (n_hi >= 0 and len(vals) > n_hi):
            raise BodyError("arity", "(%s ...) takes %s arguments, got %d"
                            % (head, n_lo if n_lo == n_hi else "%d or more" % n_lo, len(vals)))

    if head in ("+", "*", "-", "/"):
        arity(1, -1)
        if len(vals) == 1:
            v = vals[0]
            if _is_num(v):
                return {"+": v, "*": v, "-": -v}.get(head) if head != "/" else _NUMBER_BINARY["/"](1.0, v)
            t = _f32(v, L, head)
            if head == "-":
                return np.negative(t)
            return _div(np.float32(1.0), t) if head == "/" else t
        acc = vals[0]
        for v in vals[1:]:
            if _is_num(acc) and _is_num(v):
                acc = _NUMBER_BINARY[head](acc, v)
            else:
                a, b = _f32(acc, L, head), _f32(v, L, head)
                _widths_fit([a, b], head)
                acc = _TENSOR_BINARY[head](a, b)
        return acc
    if head in _COMPARE:
        arity(2)
        a, b = vals
        if _is_num(a) and _is_num(b):
            return _NUMBER_COMPARE[head](a, b)
        a, b = _f32(a, L, head), _f32(b, L, head)
        _widths_fit([a, b], head)
        return _COMPARE[head](a, b)
    if head in ("and", "or"):
        arity(1, -1)
        ts = [_bool(v, L, head) for v in vals]
        _widths_fit(ts, head)
        acc = ts[0]
        for t in ts[1:]:
            acc = (acc & t) if head == "and" else (acc | t)
        return acc
    if head == "not":
        arity(1)
        return ~_bool(vals[0], L, "not")
    if head == "where":
        arity(3)
        m = _bool(vals[0], L, "where mask")
        a, b = (_as_tensor(v, L) for v in vals[1:])
        if a.dtype != b.dtype:
            raise BodyError("E-DIM-002", "where: branches of different dtypes")
        _widths_fit([m, a, b], "where")
        return np.where(m, a, b)
    if head in ("neg", "abs"):
        arity(1)
        t = _f32(vals[0], L, head)
        return np.negative(t) if head == "neg" else np.abs(t)
    if head == "sqrt":
        arity(1)
        if _is_num(vals[0]):
            x = vals[0]
            return math.sqrt(x) if x >= 0 else math.nan
        with np.errstate(all="ignore"):
            return np.sqrt(_f32(vals[0], L, "sqrt"))
    if head in _UNARY_F64:
        arity(1)
        if head in _NUMBER_UNARY and _is_num(vals[0]):
            with np.errstate(all="ignore"):
                return float(_UNARY_F64[head](np.float64(vals[0])))
        return _via_f64(_UNARY_F64[head], _f32(vals[0], L, head))
    if head in ("pow", "atan2", "maximum", "minimum"):
        arity(2)
        if head == "pow" and _is_num(vals[0]) and _is_num(vals[1]):
            with np.errstate(all="ignore"):
                return float(np.power(np.float64(vals[0]), np.float64(vals[1])))
        a, b = _f32(vals[0], L, head), _f32(vals[1], L, head)
        _widths_fit([a, b], head)
        if head == "pow":
            return _via_f64(np.power, a, b)
        if head == "atan2":
            return _via_f64(np.arctan2, a, b)
        a, b = np.broadcast_arrays(a, b)
        return _ieee_maximum(a, b) if head == "maximum" else _ieee_minimum(a, b)
    raise BodyError("op", "`%s` is not an operation a body may use" % head)


class Body:
    """A parsed body: argument names and the expression."""

    def __init__(self, text: str):
        form = read_sexpr(text)
        if not (isinstance(form, list) and len(form) >= 3 and form[0] == "lambda" and isinstance(form[1], list)):
            raise BodyError("parse", "a body is (lambda (h seq ...) expr)")
        params = form[1]
        if len(params) < 2 or not all(isinstance(p, Sym) for p in params):
            raise BodyError("arity", "a body takes the state and at least one sequence")
        if len(set(params)) != len(params):
            raise BodyError("arity", "repeated argument name")
        self.text = text
        self.params = list(params)
        self.exprs = form[2:]

    @property
    def n_seqs(self) -> int:
        return len(self.params) - 1

    def step(self, h, seq_values, ctx: _Ctx):
        env = {self.params[0]: h}
        for name, v in zip(self.params[1:], seq_values):
            env[name] = v
        r = None
        for e in self.exprs:
            r = _eval(e, env, ctx)
        if isinstance(r, bool) or (isinstance(r, np.ndarray) and r.dtype == np.bool_):
            raise BodyError("E-DIM-002", "the body returns bool; it must return f32")
        r = _as_tensor(r, ctx.lanes)
        if r.shape[1] != ctx.W:
            if r.shape[1] == 1 and ctx.W == 1:
                pass
            else:
                raise BodyError("E-DIM-001", "the body returns width %d; the state has width %d"
                                % (r.shape[1], ctx.W))
        return np.ascontiguousarray(np.broadcast_to(r, (ctx.lanes, ctx.W)), dtype=np.float32)

    def check(self, state_width: int, seq_widths, vector_state: bool):
        """Type-check on one lane of zeros; raises BodyError when invalid."""
        ctx = _Ctx(1, state_width, vector_state)
        h = np.zeros((1, state_width), np.float32)
        self.step(h, [np.zeros((1, w), np.float32) for w in seq_widths], ctx)


def parse_body(text: str) -> Body:
    return Body(text)


def scan_body(text, initial, seqs, axis=0, state_axis=False, reverse=False):
    """Element scan of a body given as text ("Nonlinear element scans").

    initial: sequence shape with `axis` removed; seqs: list of f32 arrays of
    one shape (with `state_axis`, the same shape except each one's last
    width, 1 or the state width).  Returns the states, the shape of the first
    full-width sequence, f32.
    """
    body = text if isinstance(text, Body) else Body(text)
    seqs = [np.ascontiguousarray(s, dtype=np.float32) for s in seqs]
    if len(seqs) != body.n_seqs:
        raise BodyError("arity", "the body takes %d sequences, got %d" % (body.n_seqs, len(seqs)))
    initial = np.asarray(initial, dtype=np.float32)
    rank = seqs[0].ndim
    ax = axis + rank if axis < 0 else axis
    if state_axis:
        W = initial.shape[-1]
        full = [s for s in seqs if s.shape[-1] == W]
        shape = list((full[0] if full else seqs[0]).shape[:-1]) + [W]
    else:
        W = 1
        shape = list(seqs[0].shape)
    O = int(np.prod(shape[:ax], dtype=np.int64))
    T = shape[ax]
    after = int(np.prod(shape[ax + 1:], dtype=np.int64))
    J = after // W
    lanes = O * J
    widths = [s.shape[-1] if state_axis else 1 for s in seqs]
    views = [s.reshape(O, T, J, w) for s, w in zip(seqs, widths)]
    ctx = _Ctx(lanes, W, state_axis)
    h = initial.reshape(lanes, W).copy()
    out = np.empty((O, T, J, W), np.float32)
    order = range(T - 1, -1, -1) if reverse else range(T)
    for t in order:
        vals = [v[:, t].reshape(lanes, w) for v, w in zip(views, widths)]
        h = body.step(h, vals, ctx)
        out[:, t] = h.reshape(O, J, W)
    return out.reshape(shape)
