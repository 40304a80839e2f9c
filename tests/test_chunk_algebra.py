"""The reading the chunked matrix-scan rests on, checked in float64 on the
CPU against the oracle's sequential scan ("matrix-scan": h[t] = a[t] @ h[t-1]
+ b[t] from zero; its gradient is the same scan run backwards on a's
transposes).

Over a chunk of trips s..e, h[e] = Phi @ h[s-1] + u[e], with Phi = a[e] ...
a[s] and u the chunk's own scan from zero; the chunks link in scan order
(carry = Phi_k @ carry + u_k) and each chunk rescanned from its carry gives
every state.  The cotangent lam[t] = a[t+1]^T lam[t+1] + g[t] is the same
recurrence in the opposite order with coefficient a[t+1]^T (the zero matrix
past the axis), so it composes the same way.  Chunks here are cut as the
library cuts them: equal lengths, the short one last in scan order."""
import numpy as np
import pytest

import oracle.matrix as M


def contractive(rng, T, n, norm=0.9):
    a = rng.standard_normal((T, n, n))
    return a / np.linalg.norm(a, ord=2, axis=(-2, -1))[:, None, None] * norm


def close(got, want):
    """The oracle scans in f32 (the kernels' arithmetic): agreement to f32
    rounding, scaled by 1 + |value|."""
    err = np.abs(got - want) / (1.0 + np.abs(want))
    assert float(err.max()) <= 1e-5, float(err.max())


def chunked_scan(coef, b, chunk):
    """h[t] = coef[t] @ h[t-1] + b[t] over axis 0 from zero, by chunks."""
    T, n = coef.shape[0], coef.shape[1]
    m = b.shape[2]
    starts = list(range(0, T, chunk))
    phis, us = [], []
    for s in starts:                                  # every chunk from zero, and its product
        phi, u = np.eye(n), np.zeros((n, m))
        for t in range(s, min(T, s + chunk)):
            phi = coef[t] @ phi
            u = coef[t] @ u + b[t]
        phis.append(phi)
        us.append(u)
    carries, carry = [], np.zeros((n, m))
    for phi, u in zip(phis, us):                      # the link, in scan order
        carries.append(carry)
        carry = phi @ carry + u
    out = np.empty((T, n, m))
    for s, c in zip(starts, carries):                 # every chunk again from its carry
        h = c
        for t in range(s, min(T, s + chunk)):
            h = coef[t] @ h + b[t]
            out[t] = h
    return out


@pytest.mark.parametrize("T,chunk", [(1000, 66), (257, 64), (64, 64), (5, 2)])
@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
def test_chunked_forward_matches_the_scan(T, chunk, reverse):
    rng = np.random.default_rng(T + chunk)
    n, m = 4, 3
    a = contractive(rng, T, n).astype(np.float32)
    b = rng.standard_normal((T, n, m)).astype(np.float32)
    want = M.matrix_scan(a[None], b[None], axis=1, reverse=reverse)[0]
    a, b = a.astype(np.float64), b.astype(np.float64)
    if reverse:      # scan order is descending t: chunk the flipped sequence
        got = chunked_scan(a[::-1], b[::-1], chunk)[::-1]
    else:
        got = chunked_scan(a, b, chunk)
    close(got, want)


@pytest.mark.parametrize("T,chunk", [(1000, 66), (257, 64), (5, 2)])
@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
def test_chunked_cotangent_matches_the_gradient(T, chunk, reverse):
    rng = np.random.default_rng(7 * T + chunk)
    n, m = 4, 3
    a = contractive(rng, T, n).astype(np.float32)
    b = rng.standard_normal((T, n, m)).astype(np.float32)
    g = rng.standard_normal((T, n, m)).astype(np.float32)
    h = M.matrix_scan(a[None], b[None], axis=1, reverse=reverse)[0]
    _, want_gb = M.matrix_scan_backward(a[None], b[None], h[None], g[None], axis=1, reverse=reverse)
    a, g = a.astype(np.float64), g.astype(np.float64)
    # the cotangent scans in the opposite order with the transposed coefficient
    # of the trip after t in the forward's order, zero past the axis
    zero = np.zeros((1, n, n))
    if not reverse:
        coef = np.concatenate([np.swapaxes(a[1:], 1, 2), zero])      # coef[t] = a[t+1]^T
        lam = chunked_scan(coef[::-1], g[::-1], chunk)[::-1]
    else:
        coef = np.concatenate([zero, np.swapaxes(a[:-1], 1, 2)])     # coef[t] = a[t-1]^T
        lam = chunked_scan(coef, g, chunk)
    close(lam, want_gb[0])
