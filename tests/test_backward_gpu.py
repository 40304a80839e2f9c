"""Backward pass on the GPU against the oracle's backward, element by element.

Both sides get the same forward states (the oracle's, or the GPU's for the
full-size runs, which are compared element by element), so the comparison
isolates the backward arithmetic.  The
backward uses no transcendental and the kernels follow the definition's
operation order (NORMCAP's sqrt and division correctly rounded), so every
gradient must match bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from element_scan_recurrences_gb300 import binding as es
from element_scan_recurrences_gb300 import workloads as wl
from parity_helpers import compare_blocks

pytestmark = pytest.mark.gpu

T_, N_, M_ = wl.TANH_DECAY, wl.NORMCAP, wl.MAXPLUS
MAXPLUS_DISTS = dict(x_dist=("uniform", -1.0, 1.0), a_dist=("uniform", 0.0, 0.1), init_dist=("uniform", -1.0, 1.0))
NORMCAP_DISTS = dict(x_dist=("normal", 0.0, 0.5), a_dist=("uniform", 0.8, 1.0), init_dist=("normal", 0.0, 0.2))


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    es.lib()
    oracle.build()
    yield
    es.set_path_override("auto")


def _bits_equal(got, want, what):
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all(), "%s: %d of %d differ; first at %s: %r vs %r" % (
        what, int((~same).sum()), same.size, np.argwhere(~same)[0], got[~same][0], want[~same][0])


def _close(got, want, what, rtol=1e-5):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    err = np.abs(got - want) / (1.0 + np.abs(want))
    assert np.all(np.isfinite(got)), what
    assert float(err.max()) <= rtol, "%s: max relative error %.3g at %s" % (what, float(err.max()),
                                                                          np.unravel_index(err.argmax(), err.shape))


def _check(w, reverse, path, exact=True):
    init, seqs = wl.make_inputs(w, "cpu")
    i_np, s_np = init.numpy(), [s.numpy() for s in seqs]
    states = oracle.scan(w.body, i_np, s_np, axis=w.axis, state_axis=w.state_axis, reverse=reverse)
    G = np.random.default_rng(7).normal(size=states.shape).astype(np.float32)
    want_i, want_s = oracle.scan_backward(w.body, i_np, s_np, states, G, axis=w.axis, state_axis=w.state_axis,
                                          reverse=reverse)
    p = es.plan_backward(w.body, w.shape, w.axis, w.shape[-1] if w.state_axis else 0,
                         w.seq_widths if w.state_axis else None, reverse)
    assert p["path"] == path, (w.name, p["path"])
    dev = "cuda"
    gi, gs = es.scan_backward(w.body, init.to(dev), [s.to(dev) for s in seqs], torch.from_numpy(states).to(dev),
                              torch.from_numpy(G).to(dev), axis=w.axis, state_axis=w.state_axis, reverse=reverse)
    es.device_status()
    cmp = _bits_equal if exact else _close
    cmp(gi.cpu().numpy(), want_i, w.name + " grad initial")
    for k in range(2):
        cmp(gs[k].cpu().numpy(), want_s[k], "%s grad seq %d" % (w.name, k))


CASES = [
    ("lane_tma", wl.custom(T_, (3, 50, 200), 1, name="tanh_lane")),
    ("lane_tma", wl.custom(T_, (2, 33, 64), 1, name="tanh_lane_T33")),
    ("lane_tma", wl.custom(M_, (2, 37, 96), 1, name="maxplus_lane", **MAXPLUS_DISTS)),
    ("lane_tma", wl.custom(M_, (4, 16, 160), 1, name="maxplus_lane_one_tile", **MAXPLUS_DISTS)),
    ("lane_tma", wl.custom(T_, (300, 40), 0, name="tanh_lane_axis0")),
    # more CTAs than SMs: the gradients go through shared-memory tiles and TMA
    # stores (ragged lane and trip tiles; 128- and 32-lane CTAs)
    ("lane_tma", wl.custom(T_, (40, 70, 1000), 1, name="tanh_lane_staged")),
    ("lane_tma", wl.custom(M_, (40, 45, 1000), 1, name="maxplus_lane_staged", **MAXPLUS_DISTS)),
    ("lane_tma", wl.custom(T_, (200, 37, 40), 1, name="tanh_lane_staged_32")),
    ("lane_tma", wl.custom(M_, (150, 40, 100), 1, name="maxplus_lane_staged_64", **MAXPLUS_DISTS)),
    ("lane_tma", wl.custom(T_, (4, 19, 8, 16), 1, state_axis=True, seq_widths=(16, 16), name="tanh_vec_full")),
    ("generic", wl.custom(T_, (5, 7, 3), 0, name="tanh_generic")),
    ("generic", wl.custom(M_, (5, 7, 3), 2, name="maxplus_generic", **MAXPLUS_DISTS)),
    ("time_tma", wl.custom(T_, (70, 64), -1, name="tanh_time_inner")),
    ("time_tma", wl.custom(T_, (130, 100), -1, name="tanh_time_ragged")),
    ("time_tma", wl.custom(M_, (70, 96), 1, name="maxplus_time", **MAXPLUS_DISTS)),
    ("time_tma", wl.custom(M_, (65, 68), -1, name="maxplus_time_ragged", **MAXPLUS_DISTS)),
    ("time_tma", wl.custom(T_, (2, 3, 128), 2, name="tanh_time_rank3")),
    ("generic", wl.custom(T_, (70, 36), -1, name="tanh_time_short")),
    ("generic", wl.custom(N_, (3, 30, 7, 16), 1, True, (16, 1), name="normcap_w16", **NORMCAP_DISTS)),
    ("generic", wl.custom(N_, (2, 25, 5, 4), 1, True, (4, 4), name="normcap_w4_fullgate", **NORMCAP_DISTS)),
    ("generic", wl.custom(N_, (2, 9, 3, 5), 1, True, (1, 5), name="normcap_bcast_x", **NORMCAP_DISTS)),
    ("generic", wl.custom(T_, (4, 11, 6, 3), 1, True, (3, 1), name="tanh_vec_gate")),
    ("generic", wl.custom(T_, (6, 1, 10), 1, name="tanh_T1")),
]


@pytest.mark.parametrize("path,w", CASES, ids=[w.name for _, w in CASES])
@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
def test_backward_matches_oracle_bitwise(path, w, reverse):
    _check(w, reverse, path)


VEC_CASES = [
    wl.custom(N_, (3, 40, 24, 16), 1, True, (16, 1), name="normcap_vec_w16", **NORMCAP_DISTS),
    wl.custom(N_, (2, 35, 40, 8), 1, True, (8, 8), name="normcap_vec_w8_fullgate", **NORMCAP_DISTS),
    wl.custom(N_, (2, 21, 64, 4), 1, True, (4, 1), name="normcap_vec_w4", **NORMCAP_DISTS),
    wl.custom(N_, (1, 17, 128, 2), 1, True, (2, 2), name="normcap_vec_w2", **NORMCAP_DISTS),
    wl.custom(N_, (33, 3, 16, 16), 0, True, (16, 1), name="normcap_vec_axis0", **NORMCAP_DISTS),
]


@pytest.mark.parametrize("w", VEC_CASES, ids=[w.name for w in VEC_CASES])
@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
def test_vector_backward_within_tolerance(w, reverse):
    """The vector-state backward kernel sums over a lane pairwise and across
    threads and multiplies by a reciprocal: within 1e-5 * (1 + |oracle|)."""
    _check(w, reverse, "vec_tma", exact=False)


@pytest.mark.parametrize("path,w", [c for c in CASES if c[0] == "lane_tma"],
                         ids=[w.name for p, w in CASES if p == "lane_tma"])
def test_generic_backward_agrees_on_lane_shapes(path, w):
    try:
        es.set_path_override("generic")
        _check(w, True, "generic")
    finally:
        es.set_path_override("auto")


def test_maxplus_backward_with_ties():
    """Tie-heavy MAXPLUS inputs: every path splits tied cotangents evenly."""
    rng = np.random.default_rng(3)
    shape = (2, 40, 64)
    x = rng.choice(np.array([-1.0, 0.0, 0.5, 1.0], np.float32), size=shape).astype(np.float32)
    c = rng.choice(np.array([0.0, 0.5], np.float32), size=shape).astype(np.float32)
    init = rng.choice(np.array([0.0, 0.5], np.float32), size=(2, 64)).astype(np.float32)
    for reverse in (False, True):
        states = oracle.scan(M_, init, [x, c], axis=1, reverse=reverse)
        G = rng.choice(np.array([1.0, -2.0, 0.75], np.float32), size=shape).astype(np.float32)
        want_i, want_s = oracle.scan_backward(M_, init, [x, c], states, G, axis=1, reverse=reverse)
        for path in ("lane_tma", "generic"):
            try:
                es.set_path_override(path)
                gi, gs = es.scan_backward(M_, torch.from_numpy(init).cuda(),
                                          [torch.from_numpy(x).cuda(), torch.from_numpy(c).cuda()],
                                          torch.from_numpy(states).cuda(), torch.from_numpy(G).cuda(), axis=1,
                                          reverse=reverse)
                es.device_status()
            finally:
                es.set_path_override("auto")
            _bits_equal(gi.cpu().numpy(), want_i, path + " ties grad initial")
            _bits_equal(gs[0].cpu().numpy(), want_s[0], path + " ties grad x")
            _bits_equal(gs[1].cpu().numpy(), want_s[1], path + " ties grad c")


@pytest.mark.parametrize("name", ["tanh_decay_lanes", "maxplus_reverse", "normcap_vector", "tanh_decay_time_inner"])
def test_full_size_backward_every_element(name):
    """Full-size backward from the GPU's own forward states, every gradient
    value against the oracle's backward (run on all host cores) of the same
    states and output gradient: bit for bit on the scalar-state kernels,
    within 1e-5 * (1 + |oracle|) on the vector-state kernel."""
    w = wl.WORKLOADS[name]
    init, seqs = wl.make_inputs(w, "cuda")
    for reverse in w.reverse:
        states = es.scan(w.body, init, seqs, axis=w.axis, state_axis=w.state_axis, reverse=reverse)
        gen = torch.Generator(device="cuda")
        gen.manual_seed(11)
        G = torch.randn(states.shape, generator=gen, device="cuda")
        gi, gs = es.scan_backward(w.body, init, seqs, states, G, axis=w.axis, state_axis=w.state_axis,
                                  reverse=reverse)
        es.device_status()
        h = lambda t: t.cpu().numpy()
        want_i, want_s = oracle.scan_backward_threads(w.body, h(init), [h(s) for s in seqs], h(states), h(G),
                                                      axis=w.axis, state_axis=w.state_axis, reverse=reverse)
        del states, G
        exact = not w.state_axis
        what = "%s reverse=%s" % (name, reverse)
        compare_blocks(w.body, h(gi), want_i, what + " grad initial", exact=exact)
        compare_blocks(w.body, h(gs[0]), want_s[0], what + " grad x", exact=exact)
        compare_blocks(w.body, h(gs[1]), want_s[1], what + " grad second", exact=exact)
        del gi, gs, want_i, want_s
        torch.cuda.empty_cache()
