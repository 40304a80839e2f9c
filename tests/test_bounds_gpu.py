"""Guard regions around every buffer a call writes (and reads): each output,
gradient and workspace is a view into a larger allocation whose margins hold a
sentinel bit pattern, and so is every input.  After each call on ragged lane
and trip tiles, forward and backward, on every kernel path:

- no word of any margin has changed (no write before or after a buffer);
- no output value still holds the sentinel (every position was written);
- no input changed;
- the result equals the same call on plain, unguarded buffers, bit for bit.

An element scan's outputs are new values of exactly the sequence shape
("Nonlinear element scans", "Arguments and body"), so a kernel may write
nothing outside them.  This is the check of out-of-bounds writes; every case
here is an ordinary in-bounds call.
"""
import math

import numpy as np
import pytest
import torch

from element_scan_recurrences_gb300 import binding as es
from element_scan_recurrences_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SENT32 = 0x7FA5A5A5        # a NaN pattern no kernel produces
SENT8 = 0xA5
PAD = 4096                 # margin on each side, in elements (keeps 16 KB alignment for f32 and i32)

T_, N_, M_ = wl.TANH_DECAY, wl.NORMCAP, wl.MAXPLUS
MAXPLUS_DISTS = dict(x_dist=("uniform", -1.0, 1.0), a_dist=("uniform", 0.0, 0.1), init_dist=("uniform", -1.0, 1.0))
NORMCAP_DISTS = dict(x_dist=("normal", 0.0, 0.5), a_dist=("uniform", 0.8, 1.0), init_dist=("normal", 0.0, 0.2))


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    es.lib()
    yield
    es.set_path_override("auto")


class Guard:
    """A buffer of `shape` inside an allocation with PAD sentinel elements
    before and after it (bytes for a uint8 workspace)."""

    def __init__(self, shape, dtype=torch.float32, device="cuda", pin=False, pad=PAD):
        self.n = int(math.prod(shape))
        self.pad = pad
        self.dtype = dtype
        self.buf = torch.empty(self.n + 2 * pad, dtype=dtype, device=device)
        if pin:
            self.buf = self.buf.pin_memory()
        self._bits().fill_(self._sent())
        self.t = self.buf[pad:pad + self.n].view(tuple(shape))

    def _sent(self):
        return SENT8 if self.dtype == torch.uint8 else SENT32

    def _bits(self):
        return self.buf if self.dtype == torch.uint8 else self.buf.view(torch.int32)

    @classmethod
    def of(cls, array):
        """A guarded device copy of a host array (f32 or i32)."""
        t = torch.from_numpy(np.ascontiguousarray(array))
        g = cls(t.shape, dtype=t.dtype)
        g.t.copy_(t)
        return g

    def check_margins(self, what):
        b = self._bits()
        s = self._sent()
        head = int((b[:self.pad] != s).sum())
        tail = int((b[self.pad + self.n:] != s).sum())
        assert head == 0 and tail == 0, "%s: %d elements before and %d after the buffer were written" % (
            what, head, tail)

    def check_written(self, what):
        inner = self._bits()[self.pad:self.pad + self.n]
        left = int((inner == self._sent()).sum())
        assert left == 0, "%s: %d of %d positions were never written" % (what, left, self.n)


def run_guarded(ins, out_specs, call, ws_bytes=0, what=""):
    """Call `call(inputs, outputs, workspace)` on guarded buffers and on plain
    ones; check margins, coverage, inputs and equality."""
    g_in = [Guard.of(a) for a in ins]
    g_out = [Guard(shape, dtype) for shape, dtype in out_specs]
    g_ws = Guard((ws_bytes,), torch.uint8) if ws_bytes else None
    n0 = es.launch_count()
    call([g.t for g in g_in], [g.t for g in g_out], g_ws.t if g_ws is not None else None)
    es.device_status()
    assert es.launch_count() > n0, what + ": nothing was launched"
    for k, g in enumerate(g_in):
        g.check_margins("%s input %d" % (what, k))
        assert g.t.cpu().numpy().tobytes() == np.ascontiguousarray(ins[k]).tobytes(), "%s: input %d changed" % (
            what, k)
    for k, g in enumerate(g_out):
        g.check_margins("%s output %d" % (what, k))
        g.check_written("%s output %d" % (what, k))
    if g_ws is not None:
        g_ws.check_margins(what + " workspace")
    # the same call on plain buffers gives the same bits
    p_in = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in ins]
    p_out = [torch.empty(shape, dtype=dtype, device="cuda") for shape, dtype in out_specs]
    p_ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda") if ws_bytes else None
    call(p_in, p_out, p_ws)
    es.device_status()
    for k, (g, p) in enumerate(zip(g_out, p_out)):
        a, b = g.t.cpu().numpy(), p.cpu().numpy()
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), "%s output %d differs from the plain call" % (
            what, k)
    return [g.t for g in g_out]


def with_path(path, fn):
    es.set_path_override(path)
    try:
        return fn()
    finally:
        es.set_path_override("auto")


# ---------------------------------------------------------------------------
# element scans with the fixed bodies, forward and backward

SCAN_CASES = [
    ("lane_tma", wl.custom(T_, (3, 50, 200), 1, name="tanh_lane")),
    ("lane_tma", wl.custom(M_, (2, 37, 96), 1, name="maxplus_lane", **MAXPLUS_DISTS)),
    ("lane_tma", wl.custom(T_, (40, 70, 1000), 1, name="tanh_lane_256")),
    ("lane_tma", wl.custom(M_, (40, 45, 1000), 1, name="maxplus_lane_staged", **MAXPLUS_DISTS)),
    ("lane_tma", wl.custom(T_, (200, 37, 40), 1, name="tanh_lane_staged_32")),
    ("lane_tma", wl.custom(T_, (4, 33, 8, 16), 1, state_axis=True, seq_widths=(16, 16), name="tanh_vec_full")),
    ("time_tma", wl.custom(T_, (300, 100), -1, name="tanh_time")),
    ("time_tma", wl.custom(M_, (129, 68), 1, name="maxplus_time", **MAXPLUS_DISTS)),
    ("vec_tma", wl.custom(N_, (3, 45, 20, 16), 1, True, (16, 1), name="normcap_w16", **NORMCAP_DISTS)),
    ("vec_tma", wl.custom(N_, (2, 21, 64, 4), 1, True, (4, 4), name="normcap_w4", **NORMCAP_DISTS)),
    ("generic", wl.custom(T_, (5, 7, 3), 0, name="tanh_axis0")),
    ("generic", wl.custom(M_, (5, 7, 3), 2, name="maxplus_axis2", **MAXPLUS_DISTS)),
    ("generic", wl.custom(N_, (3, 30, 7, 5), 1, True, (5, 1), name="normcap_w5", **NORMCAP_DISTS)),
]


def _scan_inputs(w):
    init, seqs = wl.make_inputs(w, "cpu")
    return init.numpy(), [s.numpy() for s in seqs]


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("path,w", SCAN_CASES, ids=[w.name for _, w in SCAN_CASES])
def test_scan_forward_and_backward_stay_in_bounds(path, w, reverse):
    init, seqs = _scan_inputs(w)
    sw = w.shape[-1] if w.state_axis else 0
    widths = w.seq_widths if w.state_axis else None
    assert es.plan(w.body, w.shape, w.axis, sw, widths, reverse)["path"] == path

    def fwd(i, o, _):
        es.scan_into(w.body, i[0], [i[1], i[2]], o[0], axis=w.axis, state_axis=w.state_axis, reverse=reverse)

    states = run_guarded([init] + seqs, [(w.shape, torch.float32)], fwd, what="%s fwd" % w.name)[0]
    states = states.cpu().numpy()
    G = np.random.default_rng(3).standard_normal(states.shape).astype(np.float32)
    assert es.plan_backward(w.body, w.shape, w.axis, sw, widths, reverse)["path"] == path

    def bwd(i, o, _):
        es.scan_backward(w.body, i[0], [i[1], i[2]], i[3], i[4], axis=w.axis, state_axis=w.state_axis,
                         reverse=reverse, grads=(o[0], [o[1], o[2]]))

    run_guarded([init] + seqs + [states, G], [(init.shape, torch.float32)] + [(s.shape, torch.float32) for s in seqs],
                bwd, what="%s bwd" % w.name)


def test_host_pipeline_stays_in_bounds():
    """es_scan_host_f32: the device buffers the caller lends and the pinned
    host output, in row pieces that overlap."""
    w = wl.custom(T_, (13, 57, 40), 1)
    init, seqs = _scan_inputs(w)
    for chunks in (1, 5):
        h_init, h_seqs = torch.from_numpy(init).pin_memory(), [torch.from_numpy(s).pin_memory() for s in seqs]
        h_out = Guard(w.shape, device="cpu", pin=True)
        d_init, d_out = Guard(init.shape), Guard(w.shape)
        d_seqs = [Guard(s.shape) for s in seqs]
        es.scan_host(w.body, h_init, h_seqs, h_out.t, (d_init.t, [g.t for g in d_seqs], d_out.t), axis=1,
                     chunks=chunks)
        torch.cuda.current_stream().synchronize()
        es.device_status()
        for g, nm in [(h_out, "host out"), (d_init, "device initial"), (d_out, "device out")] + \
                [(g, "device seq") for g in d_seqs]:
            g.check_margins("host pipeline chunks=%d %s" % (chunks, nm))
        h_out.check_written("host pipeline out")
        want = es.scan(w.body, torch.from_numpy(init).cuda(), [torch.from_numpy(s).cuda() for s in seqs], axis=1)
        assert torch.equal(h_out.t, want.cpu())


# ---------------------------------------------------------------------------
# body programs (run-time compiled skeletons), forward and backward

GATED = "(lambda (h x a g) (where (> g 0.5) (tanh (+ x (* a h))) h))"
BODY_CASES = [
    ("lane_tma", GATED, (3, 50, 200), 1, False, None),
    ("lane_tma", GATED, (40, 45, 1000), 1, False, None),
    ("time_tma", GATED, (300, 100), -1, False, None),
    ("generic", GATED, (5, 7, 3), 0, False, None),
    ("vec_tma", wl.NORMCAP_TEXT, (3, 45, 20, 16), 1, True, (16, 1)),
]


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("case", BODY_CASES, ids=["%s_%s" % (c[0], "x".join(map(str, c[2]))) for c in BODY_CASES])
def test_body_program_stays_in_bounds(case, reverse):
    path, text, shape, axis, state_axis, widths = case
    body = es.Body(text)
    n = body.n_seqs
    rng = np.random.default_rng(5)
    seq_shapes = [list(shape) for _ in range(n)]
    if state_axis:
        for k in range(n):
            seq_shapes[k][-1] = widths[k]
    seqs = [rng.uniform(0.0, 1.0, s).astype(np.float32) for s in seq_shapes]
    seqs[0] = rng.standard_normal(seq_shapes[0]).astype(np.float32)
    ax = axis % len(shape)
    init = (rng.standard_normal([d for i, d in enumerate(shape) if i != ax]) * 0.2).astype(np.float32)
    sw = shape[-1] if state_axis else 0
    assert body.plan(list(shape), axis, sw, widths, reverse)["path"] == path
    force = "generic" if path == "generic" else "auto"

    def fwd(i, o, _):
        with_path(force, lambda: body.scan_into(i[0], i[1:], o[0], axis=axis, state_axis=state_axis,
                                                reverse=reverse))

    states = run_guarded([init] + seqs, [(shape, torch.float32)], fwd, what="body %s fwd" % path)[0].cpu().numpy()
    G = rng.standard_normal(states.shape).astype(np.float32)

    def bwd(i, o, _):
        with_path(force, lambda: body.scan_backward(i[0], i[1:n + 1], i[n + 1], i[n + 2], axis=axis,
                                                    state_axis=state_axis, reverse=reverse,
                                                    grads=(o[0], o[1:])))

    run_guarded([init] + seqs + [states, G], [(init.shape, torch.float32)] + [(s.shape, torch.float32) for s in seqs],
                bwd, what="body %s bwd" % path)


# ---------------------------------------------------------------------------
# matrix-scan, linear-scan, table-scan

def _contractive(rng, lead, n, norm=0.95):
    a = rng.standard_normal(lead + (n, n))
    s = np.linalg.norm(a, ord=2, axis=(-2, -1))[..., None, None]
    return (a / s * norm).astype(np.float32)


MATRIX_CASES = [
    ("mat_tma", 8, 4, (3, 37, 21)),
    ("mat_tma", 16, 16, (2, 40, 5)),
    ("generic", 16, 40, (2, 23, 3)),
    ("generic", 5, 2, (2, 23, 3)),
]


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("path,n,m,lead", MATRIX_CASES, ids=["%s_n%dm%d" % c[:3] for c in MATRIX_CASES])
def test_matrix_scan_stays_in_bounds(path, n, m, lead, reverse):
    rng = np.random.default_rng(n * 31 + m)
    a = _contractive(rng, lead, n)
    b = rng.standard_normal(lead + (n, m)).astype(np.float32)
    force = "generic" if path == "generic" else "auto"
    if force == "auto":
        assert es.plan_matrix_scan(a.shape, b.shape, 1, reverse)["path"] == path
        assert es.plan_matrix_scan_backward(a.shape, b.shape, 1, reverse)["path"] == path

    def fwd(i, o, _):
        with_path(force, lambda: es.matrix_scan(i[0], i[1], axis=1, reverse=reverse, out=o[0]))

    h = run_guarded([a, b], [(b.shape, torch.float32)], fwd, what="matrix %s fwd" % path)[0].cpu().numpy()
    G = rng.standard_normal(h.shape).astype(np.float32)

    def bwd(i, o, _):
        with_path(force, lambda: es.matrix_scan_backward(i[0], i[1], i[2], i[3], axis=1, reverse=reverse,
                                                         grads=(o[0], o[1])))

    run_guarded([a, b, h, G], [(a.shape, torch.float32), (b.shape, torch.float32)], bwd,
                what="matrix %s bwd" % path)


CHUNK_CASES = [
    ("mat_chunked_tma", 16, 16, (3,), 3001),
    ("mat_chunked_tma", 8, 4, (2, 3), 777),
    ("mat_chunked", 4, 3, (2,), 1000),
    ("mat_chunked", 7, 2, (3,), 640),
]


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("path,n,m,lead,T", CHUNK_CASES, ids=["%s_n%dm%d" % c[:3] for c in CHUNK_CASES])
def test_chunked_matrix_scan_and_workspace_stay_in_bounds(path, n, m, lead, T, reverse):
    """The chunked scan for few long lanes writes its chunk summaries into the
    caller's workspace: nothing past the size it asked for."""
    rng = np.random.default_rng(n + m + T)
    a_lead = (lead[0], T) + lead[1:]
    a = _contractive(rng, a_lead, n, norm=0.97)
    b = rng.standard_normal(a_lead + (n, m)).astype(np.float32)
    need = es.matrix_scan_workspace(a.shape, b.shape, 1)
    assert need > 0

    def fwd(i, o, ws):
        with_path(path, lambda: es.matrix_scan_ws(i[0], i[1], ws, axis=1, reverse=reverse, out=o[0]))

    h = run_guarded([a, b], [(b.shape, torch.float32)], fwd, ws_bytes=need, what="%s fwd" % path)[0]
    h = h.cpu().numpy()
    if path != "mat_chunked_tma":
        return
    G = rng.standard_normal(h.shape).astype(np.float32)
    assert es.plan_matrix_scan_backward_ws(a.shape, b.shape, need, 1, reverse)["path"] == "mat_chunked_tma"

    def bwd(i, o, ws):
        es.matrix_scan_backward_ws(i[0], i[1], i[2], i[3], ws, axis=1, reverse=reverse, grads=(o[0], o[1]))

    run_guarded([a, b, h, G], [(a.shape, torch.float32), (b.shape, torch.float32)], bwd, ws_bytes=need,
                what="%s bwd" % path)


def test_static_scratch_entry_output_stays_in_bounds():
    rng = np.random.default_rng(2)
    a = _contractive(rng, (3, 2000), 8, norm=0.97)
    b = rng.standard_normal((3, 2000, 8, 4)).astype(np.float32)

    def fwd(i, o, _):
        es.matrix_scan_static(i[0], i[1], axis=1, out=o[0])

    run_guarded([a, b], [(b.shape, torch.float32)], fwd, what="static scratch")


LINEAR_CASES = [((3, 50, 200), 1), ((300, 100), -1), ((5, 7, 3), 0)]


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("shape,axis", LINEAR_CASES, ids=["lanes", "time_inner", "axis0"])
def test_linear_scan_stays_in_bounds(shape, axis, reverse):
    rng = np.random.default_rng(len(shape))
    a = rng.uniform(0.5, 0.99, shape).astype(np.float32)
    b = rng.standard_normal(shape).astype(np.float32)

    def fwd(i, o, _):
        es.linear_scan(i[0], i[1], axis=axis, reverse=reverse, out=o[0])

    h = run_guarded([a, b], [(shape, torch.float32)], fwd, what="linear fwd")[0].cpu().numpy()
    G = rng.standard_normal(shape).astype(np.float32)

    def bwd(i, o, _):
        es.linear_scan_backward(i[0], i[1], i[2], i[3], axis=axis, reverse=reverse, grads=(o[0], o[1]))

    run_guarded([a, b, h, G], [(shape, torch.float32), (shape, torch.float32)], bwd, what="linear bwd")


TABLE_CASES = [("time_tma", (150, 100), -1, 64, 16), ("time_tma", (70, 64), -1, 4096, 16),
               ("lane_tma", (3, 70, 200), 1, 64, 16), ("generic", (5, 7, 3), 0, 5, 3)]


@pytest.mark.parametrize("path,shape,axis,states,syms", TABLE_CASES, ids=["%s_%d" % (c[0], c[3]) for c in TABLE_CASES])
def test_table_scan_stays_in_bounds(path, shape, axis, states, syms):
    rng = np.random.default_rng(states)
    table = rng.integers(-2, states + 2, (states, syms)).astype(np.int32)
    sym = rng.integers(-1, syms + 1, shape).astype(np.int32)
    force = "generic" if path == "generic" else "auto"
    if force == "auto":
        assert es.plan_table_scan(states, syms, shape, axis)["path"] == path

    def fwd(i, o, _):
        with_path(force, lambda: es.table_scan(i[0], i[1], axis=axis, out=o[0]))

    run_guarded([table, sym], [(shape, torch.int32)], fwd, what="table %s" % path)
