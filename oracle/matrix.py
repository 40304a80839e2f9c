"""CPU oracle for `matrix-scan` and `linear-scan` -- TEST INFRASTRUCTURE.

Like the rest of this package, only the test suite, ``__graft_entry__.smoke()``
and the bench's CPU-baseline and reference arms may import it; it shares no
code with the CUDA library.

What it computes ("Tensor operations", operations table row `matrix-scan` and
the section "matrix-scan"):

    h[t] = a[t] @ h[t-1] + b[t]     along `axis`, from h = 0

with ``a`` of shape lead_a + [n, n] and ``b`` of shape lead_b + [n, m]; the
leading shapes broadcast NumPy-style to one shape and `axis` counts among
the leading dims (-1 is the one before the matrices).  ``reverse`` runs the
trips from the last position: h[t] = a[t] @ h[t+1] + b[t] from h[T] = 0.
The result has the broadcast leading shape + [n, m].  `linear-scan` is the
same over one-by-one matrices, with a and b broadcast to one shape
("matrix-scan" section, last paragraph of the recurrence).

``projective`` (same section): the running product of a, from the identity,
is divided by its largest magnitude after every step, and h by the same
number:

    P = a[t] @ P;  s = max |P|;  P = P / s;  h = (a[t] @ h + b[t]) / s.

Readings where the pages leave a step open (also listed with the design
notes): the computation is f32 (the table row: "computed in f32"); a matrix
product is the plain definition, each product and each sum rounded, the
terms added in the order j = 0..n-1, then b added; the division by s is
an IEEE f32 division.

Gradients (same section: "its gradient is the same scan run backwards on
a's transposes"; a projective scan "has no gradient"): with g[t] the
gradient of the states, the cotangent of h[t] is

    lam[t] = a[t+1]^T @ lam[t+1] + g[t]       (a reverse scan: a[t-1], lam[t-1])

run from zero in the opposite trip order (past the last trip the
coefficient is the zero matrix), so db[t] = lam[t] and
da[t] = lam[t] @ h[t-1]^T (h before the scan's first trip is zero).  Each
product is the plain definition in f32: a^T's rows in order j, then g
added; da[i][j] = sum over k = 0..m-1 in order of lam[i][k] * h[j][k].
"""
from __future__ import annotations

import numpy as np

__all__ = ["matrix_scan", "linear_scan", "broadcast_lead", "matrix_scan_backward", "linear_scan_backward"]


def broadcast_lead(sa, sb):
    """NumPy broadcast of two leading shapes (right-aligned, equal or 1)."""
    r = max(len(sa), len(sb))
    sa = (1,) * (r - len(sa)) + tuple(sa)
    sb = (1,) * (r - len(sb)) + tuple(sb)
    out = []
    for x, y in zip(sa, sb):
        if x != y and x != 1 and y != 1:
            raise ValueError("E-DIM-001: leading shapes %s and %s do not broadcast" % (sa, sb))
        out.append(max(x, y) if min(x, y) != 0 else 0)
    return tuple(out)


def _product(a, h):
    """a @ h in f32, each product and each sum rounded, j = 0..n-1 in order.

    a: [L, n, n], h: [L, n, c] -> [L, n, c]."""
    n = a.shape[-1]
    acc = np.multiply(a[:, :, 0:1], h[:, 0:1, :], dtype=np.float32)
    for j in range(1, n):
        acc = np.add(acc, np.multiply(a[:, :, j:j + 1], h[:, j:j + 1, :], dtype=np.float32), dtype=np.float32)
    return acc


def matrix_scan(a, b, axis=0, reverse=False, projective=False):
    """matrix-scan on host arrays; returns the states, f32."""
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    if a.ndim < 2 or b.ndim < 2:
        raise ValueError("E-DIM-001: a is [..., n, n] and b [..., n, m]")
    n = a.shape[-1]
    if a.shape[-2] != n or b.shape[-2] != n:
        raise ValueError("E-DIM-001: a %s and b %s: a must be square and share n with b" % (a.shape, b.shape))
    if n > 16:
        raise ValueError("E-DIM-001: n = %d; at most 16" % n)
    m = b.shape[-1]
    lead = broadcast_lead(a.shape[:-2], b.shape[:-2])
    if len(lead) == 0:
        raise ValueError("E-DIM-001: no leading axis to scan along")
    ax = axis + len(lead) if axis < 0 else axis
    if not 0 <= ax < len(lead):
        raise ValueError("E-DIM-001: axis %d out of range for leading shape %s" % (axis, lead))
    T = lead[ax]
    if T < 1:
        raise ValueError("E-DIM-001: the scanned axis has length %d" % T)
    a = np.broadcast_to(a, lead + (n, n))
    b = np.broadcast_to(b, lead + (n, m))
    # lanes: every leading position off the axis
    am = np.moveaxis(a, ax, 0).reshape(T, -1, n, n)
    bm = np.moveaxis(b, ax, 0).reshape(T, -1, n, m)
    L = am.shape[1]
    h = np.zeros((L, n, m), np.float32)
    P = np.broadcast_to(np.eye(n, dtype=np.float32), (L, n, n)).copy()
    out = np.empty((T, L, n, m), np.float32)
    order = range(T - 1, -1, -1) if reverse else range(T)
    with np.errstate(all="ignore"):
        for t in order:
            at = np.ascontiguousarray(am[t])
            h = np.add(_product(at, h), bm[t], dtype=np.float32)
            if projective:
                P = _product(at, P)
                s = np.abs(P).reshape(L, -1).max(axis=1).reshape(L, 1, 1)
                P = np.divide(P, s, dtype=np.float32)
                h = np.divide(h, s, dtype=np.float32)
            out[t] = h
    moved = tuple(lead[i] for i in range(len(lead)) if i != ax)
    return np.moveaxis(out.reshape((T,) + moved + (n, m)), 0, ax)


def linear_scan(a, b, axis=0, reverse=False):
    """linear-scan: h[t] = a[t] * h[t-1] + b[t] from h = 0, a and b
    broadcast to one shape (numbers included)."""
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    shape = broadcast_lead(a.shape, b.shape)
    r = matrix_scan(np.broadcast_to(a, shape)[..., None, None], np.broadcast_to(b, shape)[..., None, None],
                    axis=axis, reverse=reverse)
    return r[..., 0, 0]


def _outer_sum(lam, hp):
    """lam @ hp^T in f32: [L, n, m] x [L, n, m] -> [L, n, n], the sum over
    k = 0..m-1 in order, each product and each sum rounded."""
    m = lam.shape[-1]
    acc = np.multiply(lam[:, :, None, 0], hp[:, None, :, 0], dtype=np.float32)
    for k in range(1, m):
        acc = np.add(acc, np.multiply(lam[:, :, None, k], hp[:, None, :, k], dtype=np.float32), dtype=np.float32)
    return acc


def matrix_scan_backward(a, b, states, grad_out, axis=0, reverse=False, projective=False):
    """Gradients of sum(grad_out * matrix_scan(a, b)) with respect to a and b,
    from the forward states.  a and b have one leading shape (a broadcast
    operand's gradient is the caller's sum).  Returns (da, db), f32."""
    if projective:
        raise ValueError("E-ARG: a projective matrix-scan has no gradient")
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    states = np.asarray(states, np.float32)
    grad_out = np.asarray(grad_out, np.float32)
    if a.ndim < 3 or b.ndim < 3 or a.shape[:-2] != b.shape[:-2]:
        raise ValueError("E-DIM-001: the backward wants a [..., n, n] and b [..., n, m] of one leading shape")
    n, m = b.shape[-2], b.shape[-1]
    if a.shape[-2:] != (n, n) or states.shape != b.shape or grad_out.shape != b.shape:
        raise ValueError("E-DIM-001: shapes do not fit")
    lead = b.shape[:-2]
    ax = axis + len(lead) if axis < 0 else axis
    if not 0 <= ax < len(lead):
        raise ValueError("E-DIM-001: axis %d out of range for leading shape %s" % (axis, lead))
    T = lead[ax]
    am = np.moveaxis(a, ax, 0).reshape(T, -1, n, n)
    hm = np.moveaxis(states, ax, 0).reshape(T, -1, n, m)
    gm = np.moveaxis(grad_out, ax, 0).reshape(T, -1, n, m)
    L = am.shape[1]
    da = np.empty((T, L, n, n), np.float32)
    db = np.empty((T, L, n, m), np.float32)
    lam = np.zeros((L, n, m), np.float32)
    zero_a = np.zeros((L, n, n), np.float32)
    zero_h = np.zeros((L, n, m), np.float32)
    # the opposite of the scan's trip order
    order = range(T) if reverse else range(T - 1, -1, -1)
    with np.errstate(all="ignore"):
        for t in order:
            tn = t - 1 if reverse else t + 1          # the trip after t in scan order
            tp = t + 1 if reverse else t - 1          # the trip before t in scan order
            aT = np.ascontiguousarray(np.swapaxes(am[tn], 1, 2)) if 0 <= tn < T else zero_a
            lam = np.add(_product(aT, lam), gm[t], dtype=np.float32)
            db[t] = lam
            hp = hm[tp] if 0 <= tp < T else zero_h
            da[t] = _outer_sum(lam, hp)
    moved = tuple(lead[i] for i in range(len(lead)) if i != ax)
    da = np.moveaxis(da.reshape((T,) + moved + (n, n)), 0, ax)
    db = np.moveaxis(db.reshape((T,) + moved + (n, m)), 0, ax)
    return da, db


def linear_scan_backward(a, b, states, grad_out, axis=0, reverse=False):
    """Gradients of a linear-scan with a and b of one shape: (da, db)."""
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    if a.shape != b.shape:
        raise ValueError("E-DIM-001: the backward wants a and b of one shape")
    da, db = matrix_scan_backward(a[..., None, None], b[..., None, None], np.asarray(states)[..., None, None],
                                  np.asarray(grad_out)[..., None, None], axis=axis, reverse=reverse)
    return da[..., 0, 0], db[..., 0, 0]
