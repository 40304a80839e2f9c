"""Pins of the matrix-scan / linear-scan oracle (``oracle.matrix``) to facts
from outside it.

Each ``pin_*`` takes the oracle module (``matrix_scan`` and ``linear_scan``)
and raises ``AssertionError`` when it disagrees with what the pages
("Tensor operations": the `matrix-scan` row and section) and plain
mathematics fix.  ``test_matrix_oracle_pins.py`` runs them on the oracle,
``test_matrix_oracle_mutations.py`` on copies with planted mistakes.

The facts:
  * a = identity turns the scan into a running sum of b (``np.add.accumulate``,
    sequential f32, bit for bit), forward and reverse;
  * a general contractive scan agrees with an f64 loop over ``np.matmul``;
    a diagonal one with the closed form sum_s (prod_r a_r) b_s;
  * the pages' delta rule with unit keys and beta = 1 stores each value under
    its key: S_t^T k_t = v_t;
  * the columns of h are independent recurrences on the shared a ("Every
    column of h is its own recurrence"), so scanning one column at a time
    gives the same bits; broadcasting a leading dim equals materialising it;
  * reverse = flip-scan-flip; the axis may sit anywhere among the leading
    dims; h[0] = b[0];
  * linear-scan against ``scipy.signal.lfilter`` and numbers broadcast;
  * projective scans: with a = c I the normalised product stays I, so
    h_t = h_{t-1} + b_t / c exactly for c a power of two; with b zero after
    its first step, h_t points along (a_t ... a_1) b_0 with a positive factor;
  * shapes the contract rejects.

Gradients ("its gradient is the same scan run backwards on a's
transposes"; a projective scan has none):
  * a = identity makes the cotangent a reverse running sum of the state
    gradients (``np.add.accumulate`` on the flipped sequence, bit for bit),
    and da[t] = db[t] h[t-1]^T against an f64 ``np.einsum``;
  * a general scan's gradients agree with PyTorch autograd of an f64 loop
    over ``torch.matmul``, forward and reverse;
  * linear-scan: the cotangent of a constant-coefficient scan is
    ``scipy.signal.lfilter`` run backwards, and da[t] is the one product
    lam[t] h[t-1];
  * reverse = flip-backward-flip, axis placement, zero state gradients give
    zero gradients; a projective scan and broadcast operands are refused.
"""
from __future__ import annotations

import numpy as np
import scipy.signal

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
    assert not bad.any(), "%s: %d of %d values differ bitwise" % (what, int(bad.sum()), bad.size)


def assert_close(got, want, tol, what=""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    err = np.abs(got - want) / (1.0 + np.abs(want))
    assert np.all(err <= tol), "%s: max scaled error %.3g > %.3g" % (what, float(err.max()), tol)


def contractive(rng, shape, n, norm=0.9):
    """Random matrices scaled to spectral norm `norm` (inputs, not arithmetic
    of the scan)."""
    a = rng.standard_normal(shape + (n, n))
    s = np.linalg.norm(a, ord=2, axis=(-2, -1))[..., None, None]
    return (a / s * norm).astype(f32)


def pin_identity_is_running_sum(M):
    rng = _rng(1)
    b = rng.standard_normal((3, 20, 4, 5)).astype(f32)
    eye = np.broadcast_to(np.eye(4, dtype=f32), (3, 20, 4, 4))
    assert_bitwise(M.matrix_scan(eye, b, axis=1), np.add.accumulate(b, axis=1, dtype=f32), "identity")
    want = np.add.accumulate(b[:, ::-1], axis=1, dtype=f32)[:, ::-1]
    assert_bitwise(M.matrix_scan(eye, b, axis=1, reverse=True), want, "identity reverse")


def pin_matches_f64_matmul_loop(M):
    rng = _rng(2)
    for n, m in ((3, 2), (16, 16), (8, 1), (1, 4)):
        a = contractive(rng, (2, 30), n)
        b = rng.standard_normal((2, 30, n, m)).astype(f32)
        h = np.zeros((2, n, m))
        want = np.empty((2, 30, n, m))
        for t in range(30):
            h = np.matmul(a[:, t].astype(np.float64), h) + b[:, t]
            want[:, t] = h
        assert_close(M.matrix_scan(a, b, axis=1), want, 1e-5, "n=%d m=%d" % (n, m))
    # diagonal a: the closed form sum_s (prod_{r=s+1..t} a_r) b_s per entry
    d = rng.uniform(0.5, 1.0, (40, 3)).astype(f32)
    a = np.zeros((40, 3, 3), f32)
    a[:, np.arange(3), np.arange(3)] = d
    b = rng.standard_normal((40, 3, 2)).astype(f32)
    got = M.matrix_scan(a, b, axis=0).astype(np.float64)
    dd = d.astype(np.float64)
    for t in (0, 7, 39):
        want = sum(np.prod(dd[s + 1:t + 1], axis=0)[:, None] * b[s] for s in range(t + 1))
        assert_close(got[t], want, 1e-5, "diagonal t=%d" % t)


def pin_delta_rule_stores_values(M):
    """The pages' delta rule S_t = (I - beta k k^T) S_{t-1} + beta k v^T
    with unit keys and beta = 1: reading key k_t back gives v_t."""
    rng = _rng(3)
    n, m, T = 8, 5, 12
    k = rng.standard_normal((T, n))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, m))
    a = (np.eye(n) - k[:, :, None] * k[:, None, :]).astype(f32)
    b = (k[:, :, None] * v[:, None, :]).astype(f32)
    S = M.matrix_scan(a, b, axis=0).astype(np.float64)
    for t in range(T):
        assert np.allclose(S[t].T @ k[t], v[t], atol=2e-5), t


def pin_columns_and_broadcast(M):
    rng = _rng(4)
    a = contractive(rng, (2, 25), 6)
    b = rng.standard_normal((2, 25, 6, 4)).astype(f32)
    full = M.matrix_scan(a, b, axis=1)
    for k in range(4):
        assert_bitwise(M.matrix_scan(a, b[..., k:k + 1], axis=1), full[..., k:k + 1], "column %d" % k)
    # a shared by every batch row (leading dim 1) equals the materialised a
    a1 = a[:1]
    assert_bitwise(M.matrix_scan(a1, b, axis=1), M.matrix_scan(np.broadcast_to(a1, a.shape).copy(), b, axis=1),
                   "broadcast a")
    # a constant over time
    a0 = a[:, :1]
    assert_bitwise(M.matrix_scan(a0, b, axis=1),
                   M.matrix_scan(np.broadcast_to(a0, a.shape).copy(), b, axis=1), "a constant in time")
    # b broadcast over the batch
    b1 = b[:1]
    assert_bitwise(M.matrix_scan(a, b1, axis=1),
                   M.matrix_scan(a, np.broadcast_to(b1, b.shape).copy(), axis=1), "broadcast b")


def pin_structure(M):
    rng = _rng(5)
    a = contractive(rng, (3, 17, 2), 4)
    b = rng.standard_normal((3, 17, 2, 4, 3)).astype(f32)
    fwd = M.matrix_scan(a, b, axis=1)
    rev = M.matrix_scan(a, b, axis=1, reverse=True)
    assert_bitwise(rev, M.matrix_scan(a[:, ::-1], b[:, ::-1], axis=1)[:, ::-1], "reverse = flip scan flip")
    # the axis among the leading dims: -2 is axis 1 here; moving it first gives the same
    assert_bitwise(M.matrix_scan(a, b, axis=-2), fwd, "negative axis")
    moved = M.matrix_scan(np.moveaxis(a, 1, 0), np.moveaxis(b, 1, 0), axis=0)
    assert_bitwise(np.moveaxis(moved, 0, 1), fwd, "axis placement")
    # h[0] = b[0] (h starts at zero)
    bp = np.abs(b) + f32(0.5)
    assert_bitwise(M.matrix_scan(a, bp, axis=1)[:, 0], bp[:, 0], "h[0] = b[0]")


def pin_linear_scan(M):
    rng = _rng(6)
    x = rng.standard_normal((3, 200)).astype(f32)
    got = M.linear_scan(f32(0.9), x, axis=1)
    want = scipy.signal.lfilter([1.0], [1.0, -float(f32(0.9))], x.astype(np.float64), axis=1)
    assert_close(got, want, 1e-5, "constant a (a number)")
    a = rng.uniform(0.5, 1.0, (3, 60)).astype(f32)
    got = M.linear_scan(a, x[:, :60], axis=1).astype(np.float64)
    aa = a.astype(np.float64)
    for t in (0, 1, 30, 59):
        want = sum(np.prod(aa[:, s + 1:t + 1], axis=1) * x[:, s] for s in range(t + 1))
        assert_close(got[:, t], want, 1e-5, "time-varying t=%d" % t)
    # cumsum: a = 1 ("cumsum ... is built on that")
    assert_bitwise(M.linear_scan(f32(1.0), x, axis=1), np.add.accumulate(x, axis=1, dtype=f32), "cumsum")
    assert_bitwise(M.linear_scan(f32(1.0), x, axis=1, reverse=True),
                   np.add.accumulate(x[:, ::-1], axis=1, dtype=f32)[:, ::-1], "reverse cumsum")


def pin_projective(M):
    rng = _rng(7)
    n, m, T = 3, 2, 30
    # a = c I: the normalised product is I, so h_t = h_{t-1} + b_t / c exactly
    b = (rng.integers(-8, 9, (T, n, m)) / 8.0).astype(f32)
    for c in (2.0, 0.5, 4.0):
        a = np.broadcast_to(np.eye(n, dtype=f32) * f32(c), (T, n, n))
        got = M.matrix_scan(a, b, axis=0, projective=True)
        want = np.add.accumulate((b / f32(c)).astype(f32), axis=0, dtype=f32)
        assert_bitwise(got, want, "projective a = %g I" % c)
    # b zero after its first step: h_t points along (a_t ... a_1) b_0, with a positive factor
    a = (rng.standard_normal((T, n, n)) * 3).astype(f32)
    b = np.zeros((T, n, 1), f32)
    b[0] = rng.standard_normal((n, 1)).astype(f32)
    got = M.matrix_scan(a, b, axis=0, projective=True).astype(np.float64)
    v = b[0].astype(np.float64)
    for t in range(T):
        if t > 0:
            v = a[t].astype(np.float64) @ v
            v = v / np.abs(v).max()
        g = got[t][:, 0]
        assert np.all(np.isfinite(g))
        cosang = float(g @ v[:, 0]) / (np.linalg.norm(g) * np.linalg.norm(v))
        assert cosang > 1 - 1e-5, (t, cosang)
    # the normalisation follows the carried product, not each step's a: with
    # a alternating diag(2, 1), diag(1, 2) the product returns to a multiple
    # of I every second step, so s alternates 2, 1 and h alternates
    # [1/2, 1/2], [1/2, 1] (hand-derived; dyadic, so exact in f32)
    a = np.empty((8, 2, 2), f32)
    a[0::2] = np.diag([2.0, 1.0])
    a[1::2] = np.diag([1.0, 2.0])
    b = np.zeros((8, 2, 1), f32)
    b[0, :, 0] = 1.0
    want = np.empty((8, 2, 1), f32)
    want[0::2, :, 0] = [0.5, 0.5]
    want[1::2, :, 0] = [0.5, 1.0]
    assert_bitwise(M.matrix_scan(a, b, axis=0, projective=True), want, "alternating diagonal")
    # entries that would overflow f32 without the normalisation stay finite
    big = np.broadcast_to(np.array([[1e3, 1.0], [0.0, 1e3]], f32), (200, 2, 2))
    bb = np.zeros((200, 2, 1), f32)
    bb[0, :, 0] = [1.0, 1.0]
    assert np.all(np.isfinite(M.matrix_scan(big, bb, axis=0, projective=True)))
    assert not np.all(np.isfinite(M.matrix_scan(big, bb, axis=0)))


REJECTED = [
    ((4, 3, 3), (4, 3, 2), 1),          # axis out of range among the leading dims
    ((4, 3, 2), (4, 3, 2), 0),          # a not square
    ((4, 3, 3), (4, 2, 2), 0),          # n differs
    ((4, 17, 17), (4, 17, 1), 0),       # n above 16
    ((4, 3, 3), (5, 3, 1), 0),          # leading dims do not broadcast
    ((3, 3), (3, 1), 0),                # no leading axis
]


def pin_rejected_shapes(M):
    for sa, sb, axis in REJECTED:
        try:
            M.matrix_scan(np.zeros(sa, f32), np.zeros(sb, f32), axis=axis)
        except ValueError:
            continue
        raise AssertionError("accepted shapes the contract rejects: %s %s axis %d" % (sa, sb, axis))


def pin_backward_identity_is_reverse_running_sum(M):
    rng = _rng(20)
    L, T, n, m = 3, 9, 3, 2
    a = np.broadcast_to(np.eye(n, dtype=f32), (L, T, n, n)).copy()
    b = rng.standard_normal((L, T, n, m)).astype(f32)
    G = rng.standard_normal((L, T, n, m)).astype(f32)
    h = M.matrix_scan(a, b, axis=1)
    da, db = M.matrix_scan_backward(a, b, h, G, axis=1)
    want = np.flip(np.add.accumulate(np.flip(G, 1), axis=1, dtype=f32), 1)
    assert np.array_equal(_bits(db), _bits(want)), "db is not the reverse running sum of G"
    hp = np.concatenate([np.zeros_like(h[:, :1]), h[:, :-1]], axis=1).astype(np.float64)
    want_a = np.einsum("ltik,ltjk->ltij", db.astype(np.float64), hp)
    assert np.allclose(da, want_a, rtol=1e-6, atol=1e-6), "da is not db h_prev^T"
    assert not np.any(da[:, 0]), "da of the first trip (h before it is zero)"


def _torch_matrix_grads(a, b, G, axis_t, reverse):
    import torch
    ta = torch.tensor(a, dtype=torch.float64, requires_grad=True)
    tb = torch.tensor(b, dtype=torch.float64, requires_grad=True)
    T = a.shape[axis_t]
    h = torch.zeros(b.shape[0], *b.shape[2:], dtype=torch.float64)
    outs = [None] * T
    for t in (range(T - 1, -1, -1) if reverse else range(T)):
        h = ta[:, t] @ h + tb[:, t]
        outs[t] = h
    (torch.stack(outs, 1) * torch.tensor(G, dtype=torch.float64)).sum().backward()
    return ta.grad.numpy(), tb.grad.numpy()


def pin_backward_matches_autograd(M):
    rng = _rng(21)
    L, T, n, m = 2, 11, 4, 3
    a = (rng.standard_normal((L, T, n, n)) * 0.45).astype(f32)
    b = rng.standard_normal((L, T, n, m)).astype(f32)
    for reverse in (False, True):
        G = rng.standard_normal((L, T, n, m)).astype(f32)
        h = M.matrix_scan(a, b, axis=1, reverse=reverse)
        da, db = M.matrix_scan_backward(a, b, h, G, axis=1, reverse=reverse)
        wa, wb = _torch_matrix_grads(a, b, G, 1, reverse)
        for got, want, nm in ((da, wa, "da"), (db, wb, "db")):
            err = np.abs(got - want) / (1.0 + np.abs(want))
            assert float(err.max()) < 1e-5, "%s reverse=%s: %g" % (nm, reverse, float(err.max()))


def pin_backward_linear_scan(M):
    rng = _rng(22)
    T, c = 40, 0.8
    a = np.full((2, T), c, f32)
    b = rng.standard_normal((2, T)).astype(f32)
    G = rng.standard_normal((2, T)).astype(f32)
    h = M.linear_scan(a, b, axis=1)
    da, db = M.linear_scan_backward(a, b, h, G, axis=1)
    want = np.flip(scipy.signal.lfilter([1.0], [1.0, -float(f32(c))], np.flip(G.astype(np.float64), 1), axis=1), 1)
    assert np.allclose(db, want, rtol=1e-5, atol=1e-5), "linear-scan cotangent"
    hp = np.concatenate([np.zeros((2, 1), f32), h[:, :-1]], axis=1)
    assert np.array_equal(_bits(da), _bits(np.multiply(db, hp, dtype=f32))), "da[t] = lam[t] h[t-1]"


def pin_backward_structure(M):
    rng = _rng(23)
    a = (rng.standard_normal((3, 8, 2, 3, 3)) * 0.5).astype(f32)
    b = rng.standard_normal((3, 8, 2, 3, 2)).astype(f32)
    G = rng.standard_normal(b.shape).astype(f32)
    h = M.matrix_scan(a, b, axis=1)
    da, db = M.matrix_scan_backward(a, b, h, G, axis=1)
    # reverse = flip-backward-flip
    hr = M.matrix_scan(np.flip(a, 1), np.flip(b, 1), axis=1, reverse=True)
    ra, rb = M.matrix_scan_backward(np.flip(a, 1), np.flip(b, 1), hr, np.flip(G, 1), axis=1, reverse=True)
    assert np.array_equal(_bits(np.flip(ra, 1)), _bits(da)) and np.array_equal(_bits(np.flip(rb, 1)), _bits(db))
    # axis placement
    ma, mb = M.matrix_scan_backward(np.moveaxis(a, 1, 0), np.moveaxis(b, 1, 0), np.moveaxis(h, 1, 0),
                                    np.moveaxis(G, 1, 0), axis=0)
    assert np.array_equal(_bits(np.moveaxis(ma, 0, 1)), _bits(da))
    # no state gradient, no gradient
    za, zb = M.matrix_scan_backward(a, b, h, np.zeros_like(G), axis=1)
    assert not np.any(za) and not np.any(zb)
    # refused: a projective scan, broadcast operands
    for kw, aa in (({"projective": True}, a), ({}, a[:1])):
        try:
            M.matrix_scan_backward(aa, b, h, G, axis=1, **kw)
        except ValueError:
            continue
        raise AssertionError("the backward accepted %s" % kw)


ALL_PINS = [
    pin_backward_identity_is_reverse_running_sum,
    pin_backward_matches_autograd,
    pin_backward_linear_scan,
    pin_backward_structure,
    pin_identity_is_running_sum,
    pin_matches_f64_matmul_loop,
    pin_delta_rule_stores_values,
    pin_columns_and_broadcast,
    pin_structure,
    pin_linear_scan,
    pin_projective,
    pin_rejected_shapes,
]
