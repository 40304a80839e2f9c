"""matrix-scan and linear-scan gradients on the GPU against the gradient
oracle (``oracle.matrix.matrix_scan_backward``), element by element.

"matrix-scan": the gradient is the same scan run backwards on a's
transposes.  The kernels form every product in the definition's order, so
the bar is bit-identical, on the TMA and on the any-layout cotangent scan,
forward and reverse, with ragged lane and time tiles."""
import numpy as np
import pytest
import torch

import oracle.matrix as M
from element_scan_recurrences_gb300 import binding as es

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    es.lib()
    yield
    es.set_path_override("auto")


def bitwise(got, want, what):
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = got.view(np.uint32) != want.view(np.uint32)
    assert not bad.any(), "%s: %d of %d differ; first at %s: %r vs %r" % (
        what, int(bad.sum()), bad.size, np.argwhere(bad)[0], got[bad][0], want[bad][0])


def contractive(rng, lead, n):
    return (rng.standard_normal(tuple(lead) + (n, n)) * (0.9 / np.sqrt(n))).astype(np.float32)


def run_pair(a, b, axis, reverse, path, seed):
    states = M.matrix_scan(a, b, axis=axis, reverse=reverse)
    G = np.random.default_rng(seed).standard_normal(states.shape).astype(np.float32)
    want = M.matrix_scan_backward(a, b, states, G, axis=axis, reverse=reverse)
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    es.set_path_override(path)
    try:
        ga, gb = es.matrix_scan_backward(d(a), d(b), d(states), d(G), axis=axis, reverse=reverse)
        es.device_status()
    finally:
        es.set_path_override("auto")
    return (ga.cpu().numpy(), gb.cpu().numpy()), want


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("n,m", [(16, 16), (16, 4), (8, 8), (4, 3), (2, 4), (7, 2), (1, 1), (3, 5)])
@pytest.mark.parametrize("path", ["auto", "generic"])
def test_matrix_backward(n, m, reverse, path):
    rng = np.random.default_rng(n * 100 + m)
    a = contractive(rng, (3, 37, 5), n)
    b = rng.standard_normal((3, 37, 5, n, m)).astype(np.float32)
    got, want = run_pair(a, b, 1, reverse, path, n + m)
    plan = es.plan_matrix_scan_backward(a.shape, b.shape, 1, reverse)
    if path == "auto" and n in (2, 4, 8, 16) and (n * m) % 4 == 0:
        assert plan["path"] == "mat_tma", plan
    bitwise(got[1], want[1], "grad_b n=%d m=%d" % (n, m))
    bitwise(got[0], want[0], "grad_a n=%d m=%d" % (n, m))


@pytest.mark.parametrize("axis", [0, -1])
def test_matrix_backward_axes(axis):
    rng = np.random.default_rng(5)
    lead = (29, 6) if axis == 0 else (6, 29)
    a = contractive(rng, lead, 4)
    b = rng.standard_normal(lead + (4, 4)).astype(np.float32)
    for reverse in (False, True):
        got, want = run_pair(a, b, axis, reverse, "auto", 7)
        bitwise(got[0], want[0], "grad_a axis=%d" % axis)
        bitwise(got[1], want[1], "grad_b axis=%d" % axis)


@pytest.mark.parametrize("T", [1, 2, 65])
def test_matrix_backward_trip_counts(T):
    rng = np.random.default_rng(T)
    a = contractive(rng, (2, T, 33), 16)
    b = rng.standard_normal((2, T, 33, 16, 16)).astype(np.float32)
    for reverse in (False, True):
        got, want = run_pair(a, b, 1, reverse, "auto", T)
        bitwise(got[0], want[0], "grad_a T=%d" % T)
        bitwise(got[1], want[1], "grad_b T=%d" % T)


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("n,m,lead", [(16, 16, (2, 1000, 3)), (4, 4, (3, 300, 2)), (8, 8, (1, 777, 5)),
                                      (16, 4, (2, 256, 4))])
def test_matrix_backward_windows(n, m, lead, reverse):
    """Enough trips that the gradient runs in windows of trips (the scan
    windows started from the states their neighbours left, the grad_a windows
    on the library's second stream): the same bits as the gradient oracle,
    with ragged last windows."""
    rng = np.random.default_rng(n * 7 + lead[1])
    a = contractive(rng, lead, n)
    b = rng.standard_normal(tuple(lead) + (n, m)).astype(np.float32)
    assert es.plan_matrix_scan_backward(a.shape, b.shape, 1, reverse)["path"] == "mat_tma"
    got, want = run_pair(a, b, 1, reverse, "auto", 11)
    bitwise(got[0], want[0], "grad_a windows n=%d m=%d T=%d" % (n, m, lead[1]))
    bitwise(got[1], want[1], "grad_b windows n=%d m=%d T=%d" % (n, m, lead[1]))


def test_matrix_backward_windows_on_a_side_stream():
    """Work queued on the caller's stream after a windowed gradient sees all
    of it (the library's stream joins back), on a non-default stream, twice in
    a row into the same buffers."""
    rng = np.random.default_rng(5)
    lead, n, m = (2, 640, 4), 16, 16
    a = contractive(rng, lead, n)
    b = rng.standard_normal(tuple(lead) + (n, m)).astype(np.float32)
    states = M.matrix_scan(a, b, axis=1)
    G = rng.standard_normal(states.shape).astype(np.float32)
    wa, wb = M.matrix_scan_backward(a, b, states, G, axis=1)
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    da_, db_, ds_, dg_ = d(a), d(b), d(states), d(G)
    ga, gb = torch.empty_like(da_), torch.empty_like(db_)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            ga.fill_(float("nan"))
            gb.fill_(float("nan"))
            es.matrix_scan_backward(da_, db_, ds_, dg_, axis=1, grads=(ga, gb), stream=side)
            ca, cb = ga.clone(), gb.clone()        # queued on the same stream right after
    side.synchronize()
    es.device_status()
    bitwise(ca.cpu(), wa, "grad_a after the join")
    bitwise(cb.cpu(), wb, "grad_b after the join")


def test_matrix_backward_refusals():
    a = torch.rand(2, 7, 4, 4, device="cuda")
    b = torch.rand(2, 7, 4, 2, device="cuda")
    h = es.matrix_scan(a, b, axis=1)
    with pytest.raises(es.EsError) as e:
        es.matrix_scan_backward(a, b, h, h.clone(), axis=1, projective=True)
    assert e.value.status == 3
    with pytest.raises(es.EsError) as e:
        es.matrix_scan_backward(a[:1].contiguous(), b, h, h.clone(), axis=1)
    assert e.value.status == 4
    with pytest.raises(es.EsError) as e:       # a gradient written over the states
        es.matrix_scan_backward(a, b, h, h.clone(), axis=1, grads=(torch.empty_like(a), h))
    assert e.value.status == 3


@pytest.mark.parametrize("shape,axis,path", [((3, 45, 40), 1, "lane_tma"), ((150, 100), -1, "time_tma"),
                                             ((3, 45, 50), 1, "generic")])
def test_linear_backward(shape, axis, path):
    rng = np.random.default_rng(11)
    a = rng.uniform(0.5, 0.99, shape).astype(np.float32)
    b = rng.standard_normal(shape).astype(np.float32)
    assert es.plan_linear_scan_backward(shape, shape, axis)["path"] == path
    for reverse in (False, True):
        states = M.linear_scan(a, b, axis=axis, reverse=reverse)
        G = rng.standard_normal(shape).astype(np.float32)
        wa, wb = M.linear_scan_backward(a, b, states, G, axis=axis, reverse=reverse)
        d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
        ga, gb = es.linear_scan_backward(d(a), d(b), d(states), d(G), axis=axis, reverse=reverse)
        es.device_status()
        bitwise(ga.cpu(), wa, "linear grad_a %s" % path)
        bitwise(gb.cpu(), wb, "linear grad_b %s" % path)


def test_linear_scan_backward_full_size_every_element():
    """The linear-scan workload's backward at full size in the bench's launch
    configuration; every gradient against the oracle (run on every host core
    over contiguous blocks of the leading dimension), bit for bit."""
    import oracle
    from element_scan_recurrences_gb300 import workloads as wl
    w = wl.MATRIX_WORKLOADS["linear_scan_lanes"]
    a, b = wl.make_matrix_inputs(w, "cuda")
    h = es.linear_scan(a, b, axis=w.axis)
    G = torch.randn(h.shape, device="cuda", generator=torch.Generator("cuda").manual_seed(3))
    ga, gb = es.linear_scan_backward(a, b, h, G, axis=w.axis)
    es.device_status()
    ah, bh, hh, gh = a.cpu().numpy(), b.cpu().numpy(), h.cpu().numpy(), G.cpu().numpy()
    del a, b, h, G
    got_a, got_b = ga.cpu().numpy(), gb.cpu().numpy()
    del ga, gb
    want_a, want_b = np.empty_like(got_a), np.empty_like(got_b)

    def rows(lo, hi):
        want_a[lo:hi], want_b[lo:hi] = M.linear_scan_backward(ah[lo:hi], bh[lo:hi], hh[lo:hi], gh[lo:hi],
                                                              axis=w.axis)
    oracle.split_rows(rows, ah.shape[0])
    for lo in range(0, ah.shape[0], 8):
        bitwise(got_a[lo:lo + 8], want_a[lo:lo + 8], "linear grad_a rows %d.." % lo)
        bitwise(got_b[lo:lo + 8], want_b[lo:lo + 8], "linear grad_b rows %d.." % lo)


def test_delta_rule_backward_full_size_every_element():
    """The delta-rule workload's backward at full size in the bench's launch
    configuration; every gradient against the oracle (run on every host core
    over contiguous blocks of the leading dimension), bit for bit."""
    import oracle
    from element_scan_recurrences_gb300 import workloads as wl
    w = wl.MATRIX_WORKLOADS["matrix_scan_delta_rule"]
    a, b = wl.make_matrix_inputs(w, "cuda")
    h = es.matrix_scan(a, b, axis=w.axis)
    G = torch.randn(h.shape, device="cuda", generator=torch.Generator("cuda").manual_seed(3))
    ga, gb = es.matrix_scan_backward(a, b, h, G, axis=w.axis)
    es.device_status()
    ah, bh, hh, gh = a.cpu().numpy(), b.cpu().numpy(), h.cpu().numpy(), G.cpu().numpy()
    del a, b, h, G
    got_a, got_b = ga.cpu().numpy(), gb.cpu().numpy()
    del ga, gb
    want_a, want_b = np.empty_like(got_a), np.empty_like(got_b)

    def rows(lo, hi):
        want_a[lo:hi], want_b[lo:hi] = M.matrix_scan_backward(ah[lo:hi], bh[lo:hi], hh[lo:hi], gh[lo:hi],
                                                              axis=w.axis)
    oracle.split_rows(rows, w.lead[0])
    for lo in range(0, w.lead[0], 8):
        bitwise(got_a[lo:lo + 8], want_a[lo:lo + 8], "grad_a rows %d.." % lo)
        bitwise(got_b[lo:lo + 8], want_b[lo:lo + 8], "grad_b rows %d.." % lo)


def spectral(rng, lead, n, norm=0.97):
    a = rng.standard_normal(tuple(lead) + (n, n))
    s = np.linalg.norm(a, ord=2, axis=(-2, -1))[..., None, None]
    return (a / s * norm).astype(np.float32)


def close(got, want, what, tol=1e-5):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    err = np.abs(got - want) / (1.0 + np.abs(want))
    assert float(err.max()) <= tol, "%s: max scaled error %.3g" % (what, float(err.max()))


CHUNK_GRAD_CASES = [(16, 16, (3,), 3001), (16, 8, (1,), 256), (8, 4, (2, 3), 777), (4, 4, (2,), 1000),
                    (2, 2, (5,), 5000)]


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("n,m,lead,T", CHUNK_GRAD_CASES,
                         ids=["n%dm%d_%s_T%d" % (c[0], c[1], "x".join(map(str, c[2])), c[3]) for c in CHUNK_GRAD_CASES])
def test_chunked_backward(n, m, lead, T, reverse):
    """Few long lanes: the cotangent scan chunked on the TMA passes (four
    launches), within 1e-5 * (1 + |value|) of the gradient oracle and of the
    sequential gradient (the chunks reassociate the cotangent chain)."""
    rng = np.random.default_rng(n * 1000 + m * 10 + T + 1)
    a_lead = (lead[0], T) + lead[1:]
    a = spectral(rng, a_lead, n)
    b = rng.standard_normal(a_lead + (n, m)).astype(np.float32)
    states = M.matrix_scan(a, b, axis=1, reverse=reverse)
    G = rng.standard_normal(states.shape).astype(np.float32)
    want = M.matrix_scan_backward(a, b, states, G, axis=1, reverse=reverse)
    need = es.matrix_scan_workspace(a.shape, b.shape, 1)
    assert es.plan_matrix_scan_backward_ws(a.shape, b.shape, need, 1, reverse)["path"] == "mat_chunked_tma"
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    da, db, dh, dg = d(a), d(b), d(states), d(G)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    n0 = es.launch_count()
    ga, gb = es.matrix_scan_backward_ws(da, db, dh, dg, ws, axis=1, reverse=reverse)
    es.device_status()
    assert es.launch_count() - n0 == 4
    sa, sb = es.matrix_scan_backward(da, db, dh, dg, axis=1, reverse=reverse)
    es.device_status()
    what = "n=%d m=%d T=%d rev=%d" % (n, m, T, reverse)
    close(gb.cpu().numpy(), want[1], "grad_b " + what)
    close(ga.cpu().numpy(), want[0], "grad_a " + what)
    close(gb.cpu().numpy(), sb.cpu().numpy(), "grad_b vs sequential " + what)
    close(ga.cpu().numpy(), sa.cpu().numpy(), "grad_a vs sequential " + what)


def test_chunked_backward_falls_back():
    """Without enough workspace, or with operands the TMA passes do not take,
    the workspace entry is the sequential gradient, bit for bit."""
    rng = np.random.default_rng(5)
    for n, m in ((4, 4), (7, 2)):
        a = spectral(rng, (2, 700), n)
        b = rng.standard_normal((2, 700, n, m)).astype(np.float32)
        states = M.matrix_scan(a, b, axis=1)
        G = rng.standard_normal(states.shape).astype(np.float32)
        want = M.matrix_scan_backward(a, b, states, G, axis=1)
        need = es.matrix_scan_workspace(a.shape, b.shape, 1)
        ws = torch.empty(max(16, need - 16 if n == 4 else need), dtype=torch.uint8, device="cuda")
        d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
        ga, gb = es.matrix_scan_backward_ws(d(a), d(b), d(states), d(G), ws, axis=1)
        es.device_status()
        bitwise(gb.cpu().numpy(), want[1], "grad_b fallback n=%d" % n)
        bitwise(ga.cpu().numpy(), want[0], "grad_a fallback n=%d" % n)
