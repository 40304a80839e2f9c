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


def sampled_lane_parity(w: workloads.Workload, init, seqs, out, reverse: bool, n_lanes: int = 48, seed: int = 1):
    """Check sampled lanes of a full-size run against the oracle lane by lane.

    The sampled lanes always include the first and the last lane.
    """
    rng = np.random.default_rng(seed)
    x, a = seqs
    ax = w.ax
    if w.state_axis:
        # [O, T, J, W] lanes (o, j)
        O, T, J, W = (int(np.prod(w.shape[:ax])), w.T, int(np.prod(w.shape[ax + 1:-1])), w.shape[-1])
        xv = x.reshape(O, T, J, W)
        av = a.reshape(O, T, J, w.seq_widths[1])
        ov = out.reshape(O, T, J, W)
        iv = init.reshape(O, J, W)
        lanes = [(0, 0), (O - 1, J - 1)] + [(int(rng.integers(O)), int(rng.integers(J))) for _ in range(n_lanes - 2)]
        oi = torch.tensor([l[0] for l in lanes], device=x.device)
        ji = torch.tensor([l[1] for l in lanes], device=x.device)
        xs = xv[oi, :, ji, :].cpu().numpy()          # [L, T, W]
        as_ = av[oi, :, ji, :].cpu().numpy()
        ins = iv[oi, ji, :].cpu().numpy()
        got = ov[oi, :, ji, :].cpu().numpy()
        want = oracle.scan(w.body, ins, [xs, as_], axis=1, state_axis=True, reverse=reverse)
    else:
        O, T = int(np.prod(w.shape[:ax])), w.T
        I = int(np.prod(w.shape[ax + 1:]))
        xv, av, ov, iv = x.reshape(O, T, I), a.reshape(O, T, I), out.reshape(O, T, I), init.reshape(O, I)
        lanes = [(0, 0), (O - 1, I - 1)] + [(int(rng.integers(O)), int(rng.integers(I))) for _ in range(n_lanes - 2)]
        oi = torch.tensor([l[0] for l in lanes], device=x.device)
        ii = torch.tensor([l[1] for l in lanes], device=x.device)
        xs = xv[oi, :, ii].cpu().numpy()             # [L, T]
        as_ = av[oi, :, ii].cpu().numpy()
        ins = iv[oi, ii].cpu().numpy()
        got = ov[oi, :, ii].cpu().numpy()
        want = oracle.scan_lanes(w.body, ins, xs, as_, reverse=reverse)
    return compare(w.body, got, want, "%s sampled lanes reverse=%s" % (w.name, reverse))
