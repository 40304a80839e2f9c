"""matrix-scan and linear-scan on the GPU against the oracle, bit for bit: the
kernels form every product and sum in the oracle's order (products rounded,
terms added j = 0..n-1, then b), so nothing is left to a tolerance.  Cases
span several lane and trip tiles with ragged tails, broadcasts, reverse and
projective scans, on both the generic and the TMA kernel."""
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
    got = np.ascontiguousarray(got, np.float32)
    want = np.ascontiguousarray(want, np.float32)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = got.view(np.uint32) != want.view(np.uint32)
    assert not bad.any(), "%s: %d of %d values differ; first at %s: %r vs %r" % (
        what, int(bad.sum()), bad.size, np.argwhere(bad)[0], got[bad][0], want[bad][0])


def contractive(rng, shape, n, norm=0.95):
    a = rng.standard_normal(shape + (n, n))
    s = np.linalg.norm(a, ord=2, axis=(-2, -1))[..., None, None]
    return (a / s * norm).astype(np.float32)


def run(a, b, axis, reverse=False, projective=False, path="auto", expect=None):
    es.set_path_override(path)
    try:
        da, db = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
        if expect is not None:
            assert es.plan_matrix_scan(a.shape, b.shape, axis, reverse, projective)["path"] == expect
        got = es.matrix_scan(da, db, axis=axis, reverse=reverse, projective=projective)
        es.device_status()
        return got.cpu().numpy()
    finally:
        es.set_path_override("auto")


TMA_CASES = [(2, 2), (4, 1), (4, 4), (8, 4), (8, 8), (16, 1), (16, 4), (16, 16)]


@pytest.mark.parametrize("projective", [False, True], ids=["plain", "projective"])
@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("n,m", TMA_CASES, ids=["n%dm%d" % c for c in TMA_CASES])
def test_matrix_tma(n, m, reverse, projective):
    if projective and n + m > 32:
        pytest.skip("projective scans carry n + m <= 32 columns")
    rng = np.random.default_rng(n * 100 + m)
    # several lane tiles with a ragged last one, several trip tiles with a ragged last one
    O, T, J = 3, 37, 21
    a = contractive(rng, (O, T, J), n)
    if projective:
        a = (a * 3).astype(np.float32)
    b = rng.standard_normal((O, T, J, n, m)).astype(np.float32)
    got = run(a, b, 1, reverse, projective, expect="mat_tma")
    bitwise(got, M.matrix_scan(a, b, axis=1, reverse=reverse, projective=projective), "tma n=%d m=%d" % (n, m))


GENERIC_CASES = [(1, 1), (3, 5), (5, 2), (7, 7), (16, 16), (16, 40), (12, 3)]


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("n,m", GENERIC_CASES, ids=["n%dm%d" % c for c in GENERIC_CASES])
def test_matrix_generic(n, m, reverse):
    rng = np.random.default_rng(7 * n + m)
    a = contractive(rng, (2, 23, 3), n)
    b = rng.standard_normal((2, 23, 3, n, m)).astype(np.float32)
    got = run(a, b, 1, reverse, path="generic")
    bitwise(got, M.matrix_scan(a, b, axis=1, reverse=reverse), "generic n=%d m=%d" % (n, m))
    if n + m <= 32:
        ap = (a * 3).astype(np.float32)
        got = run(ap, b, 1, reverse, projective=True, path="generic")
        bitwise(got, M.matrix_scan(ap, b, axis=1, reverse=reverse, projective=True), "generic projective")


def test_matrix_broadcasts_and_axes():
    rng = np.random.default_rng(3)
    n, m = 4, 3
    b = rng.standard_normal((4, 19, 5, n, m)).astype(np.float32)
    a_full = contractive(rng, (4, 19, 5), n)
    for a, what in ((a_full[:1], "a shared by the batch"), (a_full[:, :1], "a constant in time"),
                    (a_full[0, 0], "one a for every lane and trip"), (a_full[:, :, :1], "a shared by the heads")):
        got = run(np.ascontiguousarray(a), b, 1, expect="generic")
        bitwise(got, M.matrix_scan(a, b, axis=1), what)
    # b broadcast, the axis elsewhere, negative axes
    got = run(a_full, np.ascontiguousarray(b[:1]), 1)
    bitwise(got, M.matrix_scan(a_full, b[:1], axis=1), "b shared by the batch")
    for axis in (0, 2, -1, -3):
        got = run(a_full, b, axis)
        bitwise(got, M.matrix_scan(a_full, b, axis=axis), "axis %d" % axis)


def test_delta_rule_recall():
    """The pages' delta rule through the TMA kernel: unit keys, beta = 1, so
    every written value is read back under its key."""
    rng = np.random.default_rng(4)
    B, T, n, m = 8, 64, 16, 16
    k = rng.standard_normal((B, T, n))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, m))
    a = (np.eye(n) - k[..., :, None] * k[..., None, :]).astype(np.float32)
    b = (k[..., :, None] * v[..., None, :]).astype(np.float32)
    got = run(a, b, 1, expect="mat_tma")
    bitwise(got, M.matrix_scan(a, b, axis=1), "delta rule")
    S = got.astype(np.float64)
    assert np.allclose(np.einsum("btnm,btn->btm", S, k), v, atol=5e-5)


def test_linear_scan_paths():
    rng = np.random.default_rng(5)
    a = rng.uniform(0.5, 1.0, (3, 70, 200)).astype(np.float32)
    b = rng.standard_normal((3, 70, 200)).astype(np.float32)
    da, db = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    for reverse in (False, True):
        want = M.linear_scan(a, b, axis=1, reverse=reverse)
        assert es.plan_linear_scan(a.shape, b.shape, 1, reverse)["path"] == "lane_tma"
        bitwise(es.linear_scan(da, db, axis=1, reverse=reverse).cpu().numpy(), want, "lanes innermost")
        es.set_path_override("generic")
        try:
            bitwise(es.linear_scan(da, db, axis=1, reverse=reverse).cpu().numpy(), want, "generic")
        finally:
            es.set_path_override("auto")
    # the sequence axis last
    at, bt = np.ascontiguousarray(a.reshape(600, 70)[:, :68]), np.ascontiguousarray(b.reshape(600, 70)[:, :68])
    assert es.plan_linear_scan(at.shape, bt.shape, -1)["path"] == "time_tma"
    got = es.linear_scan(torch.from_numpy(at).cuda(), torch.from_numpy(bt).cuda(), axis=-1)
    bitwise(got.cpu().numpy(), M.linear_scan(at, bt, axis=-1), "time innermost")
    # numbers and broadcasts: the generic matrix kernel
    got = es.linear_scan(0.9, db, axis=1)
    bitwise(got.cpu().numpy(), M.linear_scan(np.float32(0.9), b, axis=1), "a number")
    got = es.linear_scan(torch.from_numpy(a[:, :1]).cuda(), db, axis=1, reverse=True)
    bitwise(got.cpu().numpy(), M.linear_scan(a[:, :1], b, axis=1, reverse=True), "a constant in time")
    # cumsum
    got = es.linear_scan(1.0, db, axis=1)
    bitwise(got.cpu().numpy(), np.add.accumulate(b, axis=1, dtype=np.float32), "cumsum")
    es.device_status()


@pytest.mark.parametrize("name", ["matrix_scan_delta_rule", "linear_scan_lanes"])
def test_full_size_every_element(name):
    """The bench workloads at full size in the bench's launch configuration,
    every state against the oracle (run on every host core over contiguous
    blocks of rows), bit for bit."""
    import oracle
    from element_scan_recurrences_gb300 import workloads as wl
    w = wl.MATRIX_WORKLOADS[name]
    a, b = wl.make_matrix_inputs(w, "cuda")
    if w.kind == "linear":
        out = es.linear_scan(a, b, axis=w.axis)
    else:
        out = es.matrix_scan(a, b, axis=w.axis)
    es.device_status()
    ah, bh = a.cpu().numpy(), b.cpu().numpy()
    del a, b
    want = np.empty(tuple(out.shape), np.float32)

    def rows(lo, hi):
        if w.kind == "linear":
            want[lo:hi] = M.linear_scan(ah[lo:hi], bh[lo:hi], axis=w.axis)
        else:
            want[lo:hi] = M.matrix_scan(ah[lo:hi], bh[lo:hi], axis=w.axis)
    oracle.split_rows(rows, w.lead[0])
    got = out.cpu().numpy()
    for lo in range(0, w.lead[0], 8):
        bitwise(got[lo:lo + 8], want[lo:lo + 8], "%s rows %d.." % (name, lo))


def close(got, want, what, tol=1e-5):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    err = np.abs(got - want) / (1.0 + np.abs(want))
    assert float(err.max()) <= tol, "%s: max scaled error %.3g" % (what, float(err.max()))


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("n,m,T", [(16, 16, 3001), (4, 3, 1000), (1, 1, 5000), (7, 2, 640)])
def test_chunked_few_lanes(n, m, T, reverse):
    """Few long lanes through the workspace entry: the chunked scan (chunks of
    uneven count, the last one short), within 1e-5 * (1 + |h|) of the
    sequential oracle for non-expansive a."""
    rng = np.random.default_rng(n * 7 + m + T)
    a = contractive(rng, (3, T), n, norm=0.98)
    b = rng.standard_normal((3, T, n, m)).astype(np.float32)
    need = es.matrix_scan_workspace(a.shape, b.shape, 1)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    da, db = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    n0 = es.launch_count()
    got = es.matrix_scan_ws(da, db, ws, axis=1, reverse=reverse)
    es.device_status()
    assert es.launch_count() - n0 == 3
    close(got.cpu().numpy(), M.matrix_scan(a, b, axis=1, reverse=reverse), "chunked n=%d m=%d T=%d" % (n, m, T))


CHUNK_TMA_CASES = [
    # n, m, a's leading dims (axis 1 is T), T
    (16, 16, (3,), 3001),       # the last chunk short
    (16, 8, (1,), 256),         # four chunks of 64
    (8, 24, (2,), 2000),        # n + m = 32: pass 1 carries 32 columns
    (8, 4, (2, 3), 777),        # lanes after the axis (J = 3)
    (4, 4, (2,), 1000),
    (4, 3, (2,), 1300),
    (2, 2, (5,), 5000),
]


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("n,m,lead,T", CHUNK_TMA_CASES,
                         ids=["n%dm%d_%s_T%d" % (c[0], c[1], "x".join(map(str, c[2])), c[3]) for c in CHUNK_TMA_CASES])
def test_chunked_tma_matches_chunk_kernels(n, m, lead, T, reverse):
    """The chunked scan with its scan passes on the TMA kernel takes the same
    chunks and the same arithmetic as the direct-load chunk kernels: bit for
    bit the same states, and within 1e-5 * (1 + |h|) of the sequential oracle."""
    rng = np.random.default_rng(n * 1000 + m * 10 + T)
    a_lead = (lead[0], T) + lead[1:]
    a = contractive(rng, a_lead, n, norm=0.97)
    b = rng.standard_normal(a_lead + (n, m)).astype(np.float32)
    need = es.matrix_scan_workspace(a.shape, b.shape, 1)
    assert need > 0
    assert es.plan_matrix_scan_ws(a.shape, b.shape, need, axis=1, reverse=reverse)["path"] == "mat_chunked_tma"
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    da, db = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    got = {}
    for path in ("mat_chunked_tma", "mat_chunked"):
        es.set_path_override(path)
        try:
            ws.fill_(0xFF)          # no value may leak from an earlier call's workspace
            n0 = es.launch_count()
            got[path] = es.matrix_scan_ws(da, db, ws, axis=1, reverse=reverse).cpu().numpy()
            es.device_status()
            assert es.launch_count() - n0 == 3
        finally:
            es.set_path_override("auto")
    bitwise(got["mat_chunked_tma"], got["mat_chunked"], "chunked tma vs direct n=%d m=%d" % (n, m))
    close(got["mat_chunked_tma"], M.matrix_scan(a, b, axis=1, reverse=reverse), "chunked tma n=%d m=%d" % (n, m))


def test_chunked_fallbacks_and_broadcast():
    rng = np.random.default_rng(11)
    a = contractive(rng, (2, 700), 4)
    b = rng.standard_normal((2, 700, 4, 2)).astype(np.float32)
    da, db = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    need = es.matrix_scan_workspace(a.shape, b.shape, 1)
    # too small a workspace: the sequential kernels, bit for bit
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    got = es.matrix_scan_ws(da, db, small, axis=1)
    bitwise(got.cpu().numpy(), M.matrix_scan(a, b, axis=1), "fallback")
    # forcing the chunked path without enough workspace is refused
    es.set_path_override("mat_chunked")
    try:
        with pytest.raises(es.EsError) as e:
            es.matrix_scan_ws(da, db, small, axis=1)
        assert e.value.status == 4
    finally:
        es.set_path_override("auto")
    # a shared by the lanes (broadcast), chunked
    a1 = np.ascontiguousarray(a[:1])
    need = es.matrix_scan_workspace(a1.shape, b.shape, 1)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    got = es.matrix_scan_ws(torch.from_numpy(a1).cuda(), db, ws, axis=1)
    close(got.cpu().numpy(), M.matrix_scan(a1, b, axis=1), "broadcast a, chunked")
    # projective scans never take the chunked path
    assert es.matrix_scan_workspace(a.shape, b.shape, 1, projective=True) == 0
    es.device_status()


def test_chunked_full_size_every_lane():
    """The few-lanes bench workload at full size in the bench's launch
    configuration: every lane's whole sequence of states against the oracle
    (run on every host core, one lane a thread), within tolerance."""
    import oracle
    from element_scan_recurrences_gb300 import workloads as wl
    w = wl.MATRIX_WORKLOADS["matrix_scan_few_lanes"]
    a, b = wl.make_matrix_inputs(w, "cuda")
    ws = torch.empty(es.matrix_scan_workspace(w.a_shape, w.b_shape, w.axis), dtype=torch.uint8, device="cuda")
    out = es.matrix_scan_ws(a, b, ws, axis=w.axis)
    es.device_status()
    ah, bh = a.cpu().numpy(), b.cpu().numpy()
    want = np.empty(tuple(out.shape), np.float32)

    def rows(lo, hi):
        want[lo:hi] = M.matrix_scan(ah[lo:hi], bh[lo:hi], axis=w.axis)
    oracle.split_rows(rows, w.lead[0])
    got = out.cpu().numpy()
    for lane in range(w.lead[0]):
        close(got[lane], want[lane], "lane %d" % lane)
