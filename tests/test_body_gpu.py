"""Body programs on the GPU (kernels compiled at run time from the body text)
against the body-program oracle, element by element on seeded inputs.

Every case runs on the any-layout skeleton and on the tiled skeleton its
signature selects (lanes innermost, time innermost or vector state), forward
and reverse, at sizes spanning several tiles with ragged tails.  The bar:
bit-identical where the body uses only IEEE-exact operations and the
skeleton keeps the oracle's order of a `sum`; else within
1e-5 * (1 + |oracle|).
"""
import numpy as np
import pytest
import torch

import body_cases
from element_scan_recurrences_gb300 import binding as es
from oracle.body import scan_body

pytestmark = pytest.mark.gpu

RTOL = 1e-5


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
    assert np.all(np.isfinite(got)), what + ": non-finite output"
    err = np.abs(got.astype(np.float64) - want.astype(np.float64)) / (1.0 + np.abs(want.astype(np.float64)))
    assert float(err.max()) <= RTOL, "%s: max scaled error %.3g at %s" % (
        what, float(err.max()), np.unravel_index(err.argmax(), err.shape))


def run(c, O, T, J, axis, reverse, path, seed=0):
    initial, seqs, state_axis = body_cases.make_inputs(c, O, T, J, seed=seed, axis=axis)
    body = es.Body(c[1])
    es.set_path_override(path)
    try:
        d_init = torch.from_numpy(initial).cuda()
        d_seqs = [torch.from_numpy(s).cuda() for s in seqs]
        got = body.scan(d_init, d_seqs, axis=axis, state_axis=state_axis, reverse=reverse)
        es.device_status()
        got = got.cpu().numpy()
    finally:
        es.set_path_override("auto")
    want = scan_body(c[1], initial, seqs, axis=axis, state_axis=state_axis, reverse=reverse)
    return got, want


def tiled_path(c, O, T, J, axis):
    body = es.Body(c[1])
    W = c[2]
    if W > 0:
        shape = [O, T, J, W]
        widths = c[3]
    else:
        shape = [O, T, J] if axis == 1 else [O, J, T]
        widths = None
    return body.plan(shape, axis, W, widths)["path"]


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("cid", body_cases.CASE_IDS)
def test_body_generic_path(cid, reverse):
    c = body_cases.case(cid)
    got, want = run(c, 3, 45, 40, 1, reverse, "generic")
    compare(got, want, c[6], "%s generic reverse=%s" % (cid, reverse))


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("cid", body_cases.CASE_IDS)
def test_body_tiled_path(cid, reverse):
    """The skeleton a lane-rich shape selects: several lane tiles, a ragged
    last lane tile and a ragged last time tile."""
    c = body_cases.case(cid)
    W = c[2]
    if W > 0:
        O, T, J = 2, 70, 72
    else:
        O, T, J = 3, 70, 200
    path = tiled_path(c, O, T, J, 1)
    expected = "vec_tma" if W in (2, 4, 8, 16) else "generic" if W > 1 else "lane_tma"
    assert path == expected, (cid, path)
    got, want = run(c, O, T, J, 1, reverse, "auto")
    compare(got, want, c[7], "%s %s reverse=%s" % (cid, path, reverse))


SCALAR_IDS = [c[0] for c in body_cases.CASES if c[2] == 0]


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("cid", SCALAR_IDS)
def test_body_wide_lane_tiles(cid, reverse):
    """Rows wide and a batch deep enough for 256-lane tiles: a ragged last
    lane tile (1000 = 3 x 256 + 232) and a ragged last trip tile."""
    c = body_cases.case(cid)
    O, T, J = 40, 70, 1000
    assert tiled_path(c, O, T, J, 1) == "lane_tma"
    got, want = run(c, O, T, J, 1, reverse, "auto")
    compare(got, want, c[7], "%s wide lane tiles reverse=%s" % (cid, reverse))


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("cid", SCALAR_IDS)
def test_body_time_path(cid, reverse):
    """The sequence axis last: rows of T trips transposed through shared
    memory; a ragged last row tile and a ragged last trip tile."""
    c = body_cases.case(cid)
    O, J, T = 3, 70, 100
    assert tiled_path(c, O, T, J, 2) == "time_tma"
    got, want = run(c, O, T, J, 2, reverse, "auto")
    compare(got, want, c[7], "%s time_tma reverse=%s" % (cid, reverse))


def test_page_bodies_match_fixed_kernels():
    """The pages' TANH_DECAY and MAXPLUS bodies as text give exactly what the
    built-in kernels give (same operations, same order, same tanhf)."""
    for cid, fixed in (("tanh_decay", es.TANH_DECAY), ("maxplus", es.MAXPLUS)):
        c = body_cases.case(cid)
        initial, seqs, _ = body_cases.make_inputs(c, 4, 300, 256, seed=3)
        d_init = torch.from_numpy(initial).cuda()
        d_seqs = [torch.from_numpy(s).cuda() for s in seqs]
        for reverse in (False, True):
            a = es.Body(c[1]).scan(d_init, d_seqs, axis=1, reverse=reverse)
            b = es.scan(fixed, d_init, d_seqs, axis=1, reverse=reverse)
            assert torch.equal(a.view(torch.int32), b.view(torch.int32)), (cid, reverse)


def test_body_compiles_once_per_signature():
    c = body_cases.case("average")
    body = es.Body(c[1])
    initial, seqs, _ = body_cases.make_inputs(c, 2, 40, 64, seed=4)
    d_init = torch.from_numpy(initial).cuda()
    d_seqs = [torch.from_numpy(s).cuda() for s in seqs]
    body.scan(d_init, d_seqs, axis=1)
    n0 = es.body_compile_count()
    for _ in range(3):
        body.scan(d_init, d_seqs, axis=1)
    # a second program with the same text reuses the cached kernel
    es.Body(c[1]).scan(d_init, d_seqs, axis=1)
    torch.cuda.synchronize()
    assert es.body_compile_count() == n0


def test_body_streams_and_empty():
    c = body_cases.case("maxplus")
    body = es.Body(c[1])
    initial, seqs, _ = body_cases.make_inputs(c, 2, 33, 96, seed=5)
    d_init = torch.from_numpy(initial).cuda()
    d_seqs = [torch.from_numpy(s).cuda() for s in seqs]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        got = body.scan(d_init, d_seqs, axis=1, stream=s)
    s.synchronize()
    want = scan_body(c[1], initial, seqs, axis=1)
    compare(got.cpu().numpy(), want, True, "side stream")
    # no lanes: nothing is launched, the call succeeds
    n0 = es.launch_count()
    e_init = torch.empty((0, 96), device="cuda")
    e_seqs = [torch.empty((0, 33, 96), device="cuda") for _ in range(2)]
    out = body.scan(e_init, e_seqs, axis=1)
    assert out.shape == (0, 33, 96) and es.launch_count() == n0


def test_body_misaligned_falls_back_to_generic():
    c = body_cases.case("average")
    body = es.Body(c[1])
    initial, seqs, _ = body_cases.make_inputs(c, 2, 40, 65, seed=6)
    d_init = torch.from_numpy(initial).cuda()
    buf = torch.from_numpy(np.concatenate([np.zeros(1, np.float32), seqs[0].ravel()])).cuda()
    x = buf[1:].view(seqs[0].shape)          # 4-byte aligned, not 16
    p = body.plan(list(x.shape), 1, ptrs=[d_init.data_ptr(), x.data_ptr(), 1 << 44])
    assert p["path"] == "generic"
    got = body.scan(d_init, [x], axis=1)
    compare(got.cpu().numpy(), scan_body(c[1], initial, seqs, axis=1), True, "misaligned")


@pytest.mark.parametrize("name", ["body_tanh_decay_lanes", "body_gated_lanes", "body_normcap_vector",
                                  "body_maxplus_reverse", "body_tanh_decay_time_inner"])
def test_body_full_size_every_element(name):
    """The body workloads at full size in the bench's launch configuration:
    every output value (each direction the workload names) against the
    body-program oracle run on every host core (lanes split into contiguous
    blocks of rows), bit for bit for the IEEE-exact max-plus body and within
    1e-5 * (1 + |oracle|) otherwise, plus the bound every state of the body
    obeys."""
    import oracle
    from element_scan_recurrences_gb300 import workloads as wl
    from parity_helpers import compare_blocks
    w = wl.WORKLOADS[name]
    init, seqs = wl.make_inputs(w, "cuda")
    body = es.Body(w.text)
    exact = name == "body_maxplus_reverse"
    init_h, seqs_h = init.cpu().numpy(), [s.cpu().numpy() for s in seqs]
    for reverse in w.reverse:
        out = body.scan(init, seqs, axis=w.axis, state_axis=w.state_axis, reverse=reverse)
        es.device_status()
        want = np.empty(tuple(out.shape), np.float32)

        def rows(lo, hi):
            want[lo:hi] = scan_body(w.text, init_h[lo:hi], [s[lo:hi] for s in seqs_h], axis=w.axis,
                                    state_axis=w.state_axis, reverse=reverse)
        oracle.split_rows(rows, w.shape[0])
        compare_blocks(wl.MAXPLUS if exact else wl.TANH_DECAY, out.cpu().numpy(), want,
                       "%s reverse=%s, every element" % (name, reverse), exact=exact)
        del want
        if "tanh" in name or "gated" in name:
            assert float(out.abs().max()) <= 1.0
        if "normcap" in name:
            assert float(out.square().sum(-1).sqrt().max()) <= 1.0 + 1e-6
        del out
    es.device_status()
