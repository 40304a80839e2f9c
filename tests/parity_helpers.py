"""Shared pieces of the GPU parity tests: run one workload through the CUDA
library and through the CPU oracle on the same seeded inputs and compare.

Tolerance (the stated bar for the float bodies): every output value within
1e-5 * (1 + |oracle value|) of the oracle for TANH_DECAY and NORMCAP, and
bit-identical output for MAXPLUS.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from element_scan_recurrences_gb300 import workloads
from element_scan_recurrences_gb300 import binding as es

RTOL = 1e-5


def compare(body: int, got: np.ndarray, want: np.ndarray, what: str = ""):
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if body == workloads.MAXPLUS:
        bad = got.view(np.uint32) != want.view(np.uint32)
        assert not bad.any(), "%s: %d of %d MAXPLUS values differ bitwise; first at %s: %r vs %r" % (
            what, int(bad.sum()), bad.size, np.argwhere(bad)[0], got[bad][0], want[bad][0])
        return 0.0
    assert np.all(np.isfinite(got)), what + ": non-finite output"
    err = np.abs(got.astype(np.float64) - want.astype(np.float64)) / (1.0 + np.abs(want.astype(np.float64)))
    worst = float(err.max()) if err.size else 0.0
    assert worst <= RTOL, "%s: max relative error %.3g > %.1g at %s" % (what, worst, RTOL,
                                                                         np.unravel_index(err.argmax(), err.shape))
    return worst


def compare_blocks(body: int, got: np.ndarray, want: np.ndarray, what: str = "", exact=None,
                   block: int = 1 << 23):
    """`compare` over a whole (large) tensor, a block of the flattened arrays
    at a time so that the float64 error terms stay small.  ``exact`` forces
    (True) or waives (False) the bitwise test; by default MAXPLUS is bitwise
    and the float bodies are held to the tolerance.  Returns the worst
    relative error (0 when bitwise)."""
    got = np.ascontiguousarray(got, np.float32)
    want = np.ascontiguousarray(want, np.float32)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bitwise = (body == workloads.MAXPLUS) if exact is None else exact
    g1, w1 = got.reshape(-1), want.reshape(-1)
    worst = 0.0
    for lo in range(0, g1.size, block):
        g, wv = g1[lo:lo + block], w1[lo:lo + block]
        if bitwise:
            bad = (g.view(np.uint32) != wv.view(np.uint32)) & ~(np.isnan(g) & np.isnan(wv))
            if bad.any():
                k = int(np.argmax(bad))
                raise AssertionError("%s: %d values differ bitwise in this block; first at %s: %r vs %r" % (
                    what, int(bad.sum()), np.unravel_index(lo + k, got.shape), g[k], wv[k]))
            continue
        assert np.all(np.isfinite(g)), what + ": non-finite output"
        wd = wv.astype(np.float64)
        err = np.abs(g.astype(np.float64) - wd) / (1.0 + np.abs(wd))
        k = int(err.argmax())
        if err[k] > worst:
            worst = float(err[k])
        assert worst <= RTOL, "%s: max relative error %.3g > %.1g at %s" % (
            what, worst, RTOL, np.unravel_index(lo + k, got.shape))
    return worst


def run_gpu(w: workloads.Workload, init, seqs, reverse: bool, device="cuda"):
    init_d = init.to(device).contiguous()
    seqs_d = [s.to(device).contiguous() for s in seqs]
    out = es.scan(w.body, init_d, seqs_d, axis=w.axis, state_axis=w.state_axis, reverse=reverse)
    es.device_status()
    return out


def run_oracle(w: workloads.Workload, init, seqs, reverse: bool):
    return oracle.scan(w.body, init.cpu().numpy(), [s.cpu().numpy() for s in seqs], axis=w.axis,
                       state_axis=w.state_axis, reverse=reverse)


def check_workload(w: workloads.Workload, reverse: bool, path=None, seed=None):
    """Full-tensor parity of one (small) workload; returns the worst error."""
    init, seqs = workloads.make_inputs(w, "cpu", seed)
    if path is not None:
        shape = w.shape
        p = es.plan(w.body, shape, w.axis, shape[-1] if w.state_axis else 0,
                    w.seq_widths if w.state_axis else None, reverse)
        assert p["path"] == path, (w.name, p["path"], path)
    got = run_gpu(w, init, seqs, reverse).cpu().numpy()
    want = run_oracle(w, init, seqs, reverse)
    return compare(w.body, got, want, "%s reverse=%s" % (w.name, reverse))
