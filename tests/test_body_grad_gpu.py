"""Body-program gradients on the GPU (the backward kernel compiled at run
time from the body's generated vector-Jacobian product) against the gradient
oracle, element by element on seeded inputs.

The saved states are the oracle's forward states, so that the two backward
scans see the same inputs.  The bar: bit-identical where the body uses only
IEEE-exact operations (the backward kernel is one thread per lane, its sums
over the state in state order, as the oracle's); else within
GRAD_RTOL * (1 + |oracle|), the bound the design notes derive for the
transcendental functions' last-place differences carried over the trips.
"""
import numpy as np
import pytest
import torch

import body_cases
import body_grad_pins
from element_scan_recurrences_gb300 import binding as es
from oracle.body import scan_body
from oracle.body_grad import scan_body_backward

pytestmark = pytest.mark.gpu

GRAD_RTOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    es.lib()
    yield
    es.set_path_override("auto")


def compare(got, want, exact, what):
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if exact:
        bad = got.view(np.uint32) != want.view(np.uint32)
        assert not bad.any(), "%s: %d of %d values differ bitwise; first at %s: %r vs %r" % (
            what, int(bad.sum()), bad.size, np.argwhere(bad)[0], got[bad][0], want[bad][0])
        return
    assert np.all(np.isfinite(got)), what + ": non-finite gradient"
    err = np.abs(got.astype(np.float64) - want.astype(np.float64)) / (1.0 + np.abs(want.astype(np.float64)))
    assert float(err.max()) <= GRAD_RTOL, "%s: max scaled error %.3g at %s" % (
        what, float(err.max()), np.unravel_index(err.argmax(), err.shape))


def backward_pair(text, initial, seqs, axis, state_axis, reverse, seed, path="auto"):
    """(GPU gradients, oracle gradients) from the oracle's forward states."""
    states = scan_body(text, initial, seqs, axis=axis, state_axis=state_axis, reverse=reverse)
    G = np.random.default_rng(seed).standard_normal(states.shape).astype(np.float32)
    want = scan_body_backward(text, initial, seqs, states, G, axis=axis, state_axis=state_axis, reverse=reverse)
    body = es.Body(text)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    es.set_path_override(path)
    try:
        gi, gs = body.scan_backward(d(initial), [d(s) for s in seqs], d(states), d(G), axis=axis,
                                    state_axis=state_axis, reverse=reverse)
        es.device_status()
    finally:
        es.set_path_override("auto")
    return (gi.cpu().numpy(), [g.cpu().numpy() for g in gs]), want


def check(got, want, exact, what):
    compare(got[0], want[0], exact, what + " grad_initial")
    for k, (g, w) in enumerate(zip(got[1], want[1])):
        compare(g, w, exact, what + " grad seq %d" % k)


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("cid", body_cases.CASE_IDS)
def test_body_backward(cid, reverse):
    """Every test body on the any-layout kernel: several blocks of lanes with
    a ragged last block."""
    c = body_cases.case(cid)
    initial, seqs, state_axis = body_cases.make_inputs(c, 3, 45, 50, seed=7)
    got, want = backward_pair(c[1], initial, seqs, 1, state_axis, reverse, 11, path="generic")
    check(got, want, c[6], "%s reverse=%s" % (cid, reverse))


SCALAR_IDS = [c[0] for c in body_cases.CASES if c[2] == 0]


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("cid", SCALAR_IDS)
def test_body_backward_lane_tiles(cid, reverse):
    """Scalar-state bodies on the lanes-innermost backward: a ragged lane
    tile (40 lanes: 32 + 8) and a ragged time tile; the same operations per
    trip as the oracle, so exact bodies stay bit-identical."""
    c = body_cases.case(cid)
    initial, seqs, state_axis = body_cases.make_inputs(c, 3, 45, 40, seed=8)
    assert es.Body(c[1]).plan_backward([3, 45, 40], 1, reverse=reverse)["path"] == "lane_tma"
    got, want = backward_pair(c[1], initial, seqs, 1, state_axis, reverse, 12, path="lane_tma")
    check(got, want, c[6], "%s reverse=%s" % (cid, reverse))


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("cid", SCALAR_IDS)
def test_body_backward_time_tiles(cid, reverse):
    """Scalar-state bodies with the sequence axis last on the time-innermost
    backward: 150 rows (a ragged row tile) of 100 trips (a ragged time tile)."""
    c = body_cases.case(cid)
    initial, seqs, state_axis = body_cases.make_inputs(c, 3, 100, 50, seed=10, axis=2)
    assert es.Body(c[1]).plan_backward([3, 50, 100], 2, reverse=reverse)["path"] == "time_tma"
    got, want = backward_pair(c[1], initial, seqs, 2, state_axis, reverse, 14, path="time_tma")
    check(got, want, c[6], "%s reverse=%s" % (cid, reverse))


@pytest.mark.parametrize("T", [64, 68, 96, 260])
def test_body_backward_time_trip_counts(T):
    """Exactly two tiles, a 4-trip ragged tile, three tiles, many tiles."""
    c = body_cases.case("eight_seqs")
    initial, seqs, _ = body_cases.make_inputs(c, 2, T, 40, seed=T, axis=2)
    for reverse in (False, True):
        got, want = backward_pair(c[1], initial, seqs, 2, False, reverse, T, path="time_tma")
        check(got, want, True, "T=%d reverse=%s" % (T, reverse))


VECTOR_IDS = [c[0] for c in body_cases.CASES if c[2] in (2, 4, 8, 16)]


def _vjp_sums_over_state(text, W, widths):
    """Whether the VJP sums over the state (an explicit sum, a width-one
    operand of a wide operation, the tie count of `max`): those sums run as
    shuffle butterflies on the tiled kernel, in another order than the
    oracle's w = 0..W-1."""
    src = es.Body(text).source_backward(W, widths)
    return "group_sum" in src[src.index("static void vjp("):]


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("cid", VECTOR_IDS)
def test_body_backward_vec_tiles(cid, reverse):
    """Vector-state bodies on the vector-state backward: a ragged lane tile
    and a ragged time tile.  Bit-identical unless the VJP sums over the
    state (then within the tolerance)."""
    c = body_cases.case(cid)
    W = c[2]
    J = 128 // W * 2 + 4
    initial, seqs, state_axis = body_cases.make_inputs(c, 3, 45, J, seed=9)
    assert es.Body(c[1]).plan_backward([3, 45, J, W], 1, W, c[3], reverse=reverse)["path"] == "vec_tma"
    got, want = backward_pair(c[1], initial, seqs, 1, state_axis, reverse, 13, path="vec_tma")
    exact = c[6] and not _vjp_sums_over_state(c[1], W, c[3])
    check(got, want, exact, "%s reverse=%s" % (cid, reverse))


@pytest.mark.parametrize("T", [1, 2, 17, 200])
def test_body_backward_lane_trip_counts(T):
    """One trip (the shifted-state box entirely outside), a partial tile,
    a tile and one, and many tiles."""
    c = body_cases.case("five_seqs")
    initial, seqs, _ = body_cases.make_inputs(c, 2, T, 36, seed=T)
    for reverse in (False, True):
        got, want = backward_pair(c[1], initial, seqs, 1, False, reverse, T, path="lane_tma")
        check(got, want, True, "T=%d reverse=%s" % (T, reverse))


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("ci", range(len(body_grad_pins.AUTOGRAD_CASES)))
def test_body_backward_autograd_bodies(ci, reverse):
    case = body_grad_pins.AUTOGRAD_CASES[ci]
    text, W, widths, ranges, irng = case[0], case[2], case[3], case[4], case[5]
    c = ("ag", text, W, widths, ranges, irng, False, False)
    initial, seqs, state_axis = body_cases.make_inputs(c, 2, 33, 68, seed=ci)
    got, want = backward_pair(text, initial, seqs, 1, state_axis, reverse, 100 + ci)
    check(got, want, False, "%s reverse=%s" % (text, reverse))


def _quantised(c, O, T, J, seed):
    """Inputs on a grid of quarters: ties of maximum / minimum / max are common."""
    initial, seqs, sa = body_cases.make_inputs(c, O, T, J, seed=seed)
    q = lambda a: (np.round(a * 4) / 4).astype(np.float32)
    return q(initial), [q(s) for s in seqs], sa


TIE_BODIES = [
    ("(lambda (h x) (maximum h x))", 0, None, [(0, 1)], (0, 1)),
    ("(lambda (h x c) (minimum (- h c) x))", 0, None, [(0, 1), (0, 1)], (0, 1)),
    ("(lambda (h x) (+ (* 0.5 h) (max (+ h x) :axes [-1] :keepdims true)))", 8, [8], [(0, 1)], (0, 1)),
    ("(lambda (h x) (where (> x 0.5) (abs (- h x)) (sqrt (+ h 1))))", 0, None, [(0, 1)], (0, 1)),
    ("(lambda (h g) (+ h (broadcast-to g [4])))", 4, [1], [(0, 1)], (0, 1)),
    ("(lambda (h x) 3.0)", 0, None, [(0, 1)], (0, 1)),
]


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("ti", range(len(TIE_BODIES)))
def test_body_backward_ties_bitwise(ti, reverse):
    text, W, widths, ranges, irng = TIE_BODIES[ti]
    c = ("tie", text, W, widths, ranges, irng, True, True)
    initial, seqs, sa = _quantised(c, 2, 40, 36, ti)
    # the one-thread-per-lane kernel: its sums over the state run in state order
    got, want = backward_pair(text, initial, seqs, 1, sa, reverse, ti, path="generic")
    check(got, want, True, "%s reverse=%s" % (text, reverse))
    if W == 0:
        got, want = backward_pair(text, initial, seqs, 1, sa, reverse, ti, path="lane_tma")
        check(got, want, True, "%s reverse=%s lane tiles" % (text, reverse))


@pytest.mark.parametrize("axis", [0, -1])
def test_body_backward_axes(axis):
    """The sequence axis first and last (the canonical view's O or J is 1)."""
    c = body_cases.case("five_seqs")
    rng = np.random.default_rng(3)
    shape = (37, 21) if axis == 0 else (21, 37)
    seqs = [(rng.random(shape) * (hi - lo) + lo).astype(np.float32) for lo, hi in c[4]]
    initial = rng.random(21).astype(np.float32)
    got, want = backward_pair(c[1], initial, seqs, axis, False, False, 5)
    check(got, want, True, "five_seqs axis=%d" % axis)


def test_body_forward_then_backward():
    """The library's own forward states feed its backward (one pipeline)."""
    c = body_cases.case("gated_tanh")
    initial, seqs, sa = body_cases.make_inputs(c, 2, 64, 96, seed=1)
    body = es.Body(c[1])
    d = lambda a: torch.from_numpy(a).cuda()
    di, ds = d(initial), [d(s) for s in seqs]
    states = body.scan(di, ds, axis=1)
    G = np.random.default_rng(2).standard_normal(states.shape).astype(np.float32)
    gi, gs = body.scan_backward(di, ds, states, d(G), axis=1)
    es.device_status()
    want_states = scan_body(c[1], initial, seqs, axis=1)
    wi, ws = scan_body_backward(c[1], initial, seqs, want_states, G, axis=1)
    compare(gi.cpu().numpy(), wi, False, "grad_initial")
    for g, w in zip(gs, ws):
        compare(g.cpu().numpy(), w, False, "grad seq")


def test_body_backward_streams_and_empty():
    c = body_cases.case("average")
    body = es.Body(c[1])
    # an empty call launches nothing
    n0 = es.launch_count()
    e = torch.empty(0, 5, 3, device="cuda")
    body.scan_backward(torch.empty(0, 3, device="cuda"), [e], e.clone(), e.clone(), axis=1)
    assert es.launch_count() == n0
    # a side stream
    initial, seqs, _ = body_cases.make_inputs(c, 2, 30, 20, seed=4)
    s = torch.cuda.Stream()
    states = scan_body(c[1], initial, seqs, axis=1)
    G = np.ones(states.shape, np.float32)
    d = lambda a: torch.from_numpy(a).cuda()
    with torch.cuda.stream(s):
        di, ds, dst, dg = d(initial), [d(x) for x in seqs], d(states), d(G)
        gi, gs = body.scan_backward(di, ds, dst, dg, axis=1, stream=s)
    s.synchronize()
    wi, ws = scan_body_backward(c[1], initial, seqs, states, G, axis=1)
    compare(gi.cpu().numpy(), wi, True, "grad_initial on a side stream")
    compare(gs[0].cpu().numpy(), ws[0], True, "grad x on a side stream")


def test_body_backward_rejects_overlap_on_device():
    body = es.Body("(lambda (h x) (+ (* 0.9 h) (* 0.1 x)))")
    x = torch.rand(2, 10, 4, device="cuda")
    init = torch.rand(2, 4, device="cuda")
    states = body.scan(init, [x], axis=1)
    with pytest.raises(es.EsError) as e:
        body.scan_backward(init, [x], states, states.clone(), axis=1, grads=(torch.empty_like(init), [states]))
    assert e.value.status == 3


@pytest.mark.parametrize("name", ["body_tanh_decay_lanes", "body_normcap_vector", "body_maxplus_reverse",
                                  "body_gated_lanes", "body_tanh_decay_time_inner"])
def test_body_backward_full_size_every_element(name):
    """The backward of a body workload at full size in the bench's launch
    configuration, every gradient against the gradient oracle (run on every
    host core over contiguous blocks of the leading dimension, from the same
    saved states)."""
    import oracle
    from element_scan_recurrences_gb300 import workloads as wl
    w = wl.WORKLOADS[name]
    init, seqs = wl.make_inputs(w, "cuda")
    body = es.Body(w.text)
    reverse = w.reverse[0]
    states = body.scan(init, seqs, axis=w.axis, state_axis=w.state_axis, reverse=reverse)
    G = torch.randn(states.shape, device="cuda", generator=torch.Generator("cuda").manual_seed(5))
    gi, gs = body.scan_backward(init, seqs, states, G, axis=w.axis, state_axis=w.state_axis, reverse=reverse)
    es.device_status()
    i_h, s_h = init.cpu().numpy(), [s.cpu().numpy() for s in seqs]
    st_h, g_h = states.cpu().numpy(), G.cpu().numpy()
    del states, G, seqs
    got_i, got_s = gi.cpu().numpy(), [t.cpu().numpy() for t in gs]
    del gi, gs
    want_i = np.empty_like(got_i)
    want_s = [np.empty_like(t) for t in got_s]

    def rows(lo, hi):
        wi, ws = scan_body_backward(w.text, i_h[lo:hi], [s[lo:hi] for s in s_h], st_h[lo:hi], g_h[lo:hi],
                                    axis=w.axis, state_axis=w.state_axis, reverse=reverse)
        want_i[lo:hi] = wi
        for k in range(len(ws)):
            want_s[k][lo:hi] = ws[k]
    O = w.shape[0]
    oracle.split_rows(rows, O)
    # the vector-state kernel sums over the state in its own order
    exact = name == "body_maxplus_reverse"
    compare(got_i, want_i, exact, "%s grad_initial" % name)
    step = max(1, O // 16)
    for lo in range(0, O, step):
        for k in range(len(got_s)):
            compare(got_s[k][lo:lo + step], want_s[k][lo:lo + step], exact, "%s grad seq %d rows %d.." % (name, k, lo))
