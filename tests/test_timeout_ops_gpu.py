"""Bounded waits in the body-program, matrix-scan and table-scan pipelines:
a tile that never arrives (the producer is told on the host to skip one
load) makes the kernel give up after the wait limit, record ES_E_TIMEOUT and
return; the next call is correct.  Nothing faults or hangs the GPU."""
import numpy as np
import pytest
import torch

import body_cases
import oracle.matrix as M
import oracle.table as TS
from element_scan_recurrences_gb300 import binding as es
from oracle.body import scan_body

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def restore():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    es.set_drop_tile(-1)
    es.set_wait_limit_ns(2_000_000_000)
    es.set_path_override("auto")


def drop_then_recover(run, check):
    es.device_status()                    # a clean status word
    es.set_wait_limit_ns(20_000_000)      # 20 ms
    es.set_drop_tile(3)
    run()
    with pytest.raises(es.EsError) as ei:
        es.device_status()
    assert ei.value.status == 6           # ES_E_TIMEOUT
    es.device_status()                    # the word was cleared
    es.set_drop_tile(-1)
    es.set_wait_limit_ns(2_000_000_000)
    out = run()
    es.device_status()
    check(out)


@pytest.mark.parametrize("cid,shape,axis,path", [
    ("tanh_decay", (2, 400, 64), 1, "lane_tma"),
    ("gated_tanh", (2, 64, 400), 2, "time_tma"),
    ("normcap_w16", (2, 400, 16), 1, "vec_tma"),
])
def test_body_program_pipelines(cid, shape, axis, path):
    c = body_cases.case(cid)
    O, T, J = (shape[0], shape[1], shape[2]) if axis == 1 else (shape[0], shape[2], shape[1])
    initial, seqs, state_axis = body_cases.make_inputs(c, O, T, J, axis=axis)
    body = es.Body(c[1])
    d_init = torch.from_numpy(initial).cuda()
    d_seqs = [torch.from_numpy(s).cuda() for s in seqs]
    es.set_path_override(path)
    want = scan_body(c[1], initial, seqs, axis=axis, state_axis=state_axis)

    def check(out):
        err = np.abs(out.cpu().numpy().astype(np.float64) - want) / (1 + np.abs(want.astype(np.float64)))
        assert err.max() <= 1e-5

    drop_then_recover(lambda: body.scan(d_init, d_seqs, axis=axis, state_axis=state_axis), check)


def test_matrix_scan_pipeline():
    rng = np.random.default_rng(1)
    a = (rng.standard_normal((2, 400, 8, 4, 4)) * 0.4).astype(np.float32)
    b = rng.standard_normal((2, 400, 8, 4, 4)).astype(np.float32)
    assert es.plan_matrix_scan(a.shape, b.shape, 1)["path"] == "mat_tma"
    da, db = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    want = M.matrix_scan(a, b, axis=1)
    drop_then_recover(lambda: es.matrix_scan(da, db, axis=1),
                      lambda out: np.testing.assert_array_equal(out.cpu().numpy(), want))


def test_matrix_scan_chunked_pipeline():
    """Both TMA passes of the chunked scan give up on the missing tile; the
    next call is correct."""
    rng = np.random.default_rng(2)
    # 16 x 16 blocks: tiles of 4 trips, so a chunk (66 trips) has a tile 3
    a = (rng.standard_normal((2, 3000, 16, 16)) * 0.1).astype(np.float32)
    b = rng.standard_normal((2, 3000, 16, 16)).astype(np.float32)
    need = es.matrix_scan_workspace(a.shape, b.shape, 1)
    assert es.plan_matrix_scan_ws(a.shape, b.shape, need, axis=1)["path"] == "mat_chunked_tma"
    da, db = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    want = M.matrix_scan(a, b, axis=1)

    def check(out):
        err = np.abs(out.cpu().numpy().astype(np.float64) - want) / (1 + np.abs(want.astype(np.float64)))
        assert err.max() <= 1e-5

    drop_then_recover(lambda: es.matrix_scan_ws(da, db, ws, axis=1), check)


def test_matrix_scan_chunked_backward_pipeline():
    """The chunked cotangent scan's TMA passes give up on the missing tile;
    the next call is correct."""
    rng = np.random.default_rng(3)
    a = (rng.standard_normal((2, 3000, 16, 16)) * 0.1).astype(np.float32)
    b = rng.standard_normal((2, 3000, 16, 16)).astype(np.float32)
    h = M.matrix_scan(a, b, axis=1)
    G = rng.standard_normal(h.shape).astype(np.float32)
    wa, wb = M.matrix_scan_backward(a, b, h, G, axis=1)
    need = es.matrix_scan_workspace(a.shape, b.shape, 1)
    assert es.plan_matrix_scan_backward_ws(a.shape, b.shape, need, 1)["path"] == "mat_chunked_tma"
    da, db, dh, dg = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (a, b, h, G))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")

    def check(out):
        for got, want in zip(out, (wa, wb)):
            err = np.abs(got.cpu().numpy().astype(np.float64) - want) / (1 + np.abs(want.astype(np.float64)))
            assert err.max() <= 1e-5

    drop_then_recover(lambda: es.matrix_scan_backward_ws(da, db, dh, dg, ws, axis=1), check)


def test_matrix_scan_backward_pipeline():
    """The cotangent scan (the TMA kernel on a's transposes) gives up a
    missing tile, then recovers."""
    rng = np.random.default_rng(3)
    a = (rng.standard_normal((2, 400, 8, 4, 4)) * 0.4).astype(np.float32)
    b = rng.standard_normal((2, 400, 8, 4, 4)).astype(np.float32)
    assert es.plan_matrix_scan_backward(a.shape, b.shape, 1)["path"] == "mat_tma"
    h = M.matrix_scan(a, b, axis=1)
    G = rng.standard_normal(h.shape).astype(np.float32)
    wa, wb = M.matrix_scan_backward(a, b, h, G, axis=1)
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    da, db, dh, dg = d(a), d(b), d(h), d(G)

    def check(out):
        np.testing.assert_array_equal(out[0].cpu().numpy(), wa)
        np.testing.assert_array_equal(out[1].cpu().numpy(), wb)

    drop_then_recover(lambda: es.matrix_scan_backward(da, db, dh, dg, axis=1), check)


@pytest.mark.parametrize("shape,axis,path", [((130, 400), -1, "time_tma"), ((2, 400, 64), 1, "lane_tma")])
def test_table_scan_pipelines(shape, axis, path):
    rng = np.random.default_rng(2)
    table = rng.integers(0, 16, (16, 4)).astype(np.int32)
    sym = rng.integers(0, 4, shape).astype(np.int32)
    assert es.plan_table_scan(16, 4, shape, axis)["path"] == path
    dt, ds = torch.from_numpy(table).cuda(), torch.from_numpy(sym).cuda()
    want = TS.table_scan(table, sym, axis=axis)
    drop_then_recover(lambda: es.table_scan(dt, ds, axis=axis),
                      lambda out: np.testing.assert_array_equal(out.cpu().numpy(), want))


@pytest.mark.parametrize("path,axis", [("lane_tma", 1), ("time_tma", 2), ("vec_tma", 1)])
def test_body_backward_pipelines(path, axis):
    """Each tiled backward gives up a missing tile, then recovers."""
    from oracle.body_grad import scan_body_backward
    # a body with no sum over the state: bit-exact on every path
    c = body_cases.case("maxplus")
    if path == "vec_tma":
        c = ("maxplus_w8", c[1], 8, [8, 8]) + tuple(c[4:])
    initial, seqs, sa = body_cases.make_inputs(c, 2, 400, 64, axis=axis)
    states = scan_body(c[1], initial, seqs, axis=axis, state_axis=sa)
    G = np.random.default_rng(1).standard_normal(states.shape).astype(np.float32)
    want = scan_body_backward(c[1], initial, seqs, states, G, axis=axis, state_axis=sa)
    body = es.Body(c[1])
    d = lambda a: torch.from_numpy(a).cuda()
    di, ds, dst, dg = d(initial), [d(s) for s in seqs], d(states), d(G)
    es.set_path_override(path)

    def run():
        return body.scan_backward(di, ds, dst, dg, axis=axis, state_axis=sa)

    def check(out):
        gi, gs = out
        assert np.array_equal(gi.cpu().numpy(), want[0])
        for g, w in zip(gs, want[1]):
            assert np.array_equal(g.cpu().numpy(), w)

    drop_then_recover(run, check)
