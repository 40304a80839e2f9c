"""CUDA library vs the CPU oracle, element by element, on seeded inputs.

Small cases cover every kernel path with several tiles and ragged tails in
both directions; the five measured workloads run at full size in the launch
configuration the bench times and are checked element by element (against the
oracle on all host cores) plus properties that hold at any size.  MAXPLUS must be bit-exact; TANH_DECAY and NORMCAP within
1e-5 * (1 + |oracle|).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from element_scan_recurrences_gb300 import binding as es
from element_scan_recurrences_gb300 import workloads as wl
from parity_helpers import check_workload, compare, compare_blocks, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

T_, N_, M_ = wl.TANH_DECAY, wl.NORMCAP, wl.MAXPLUS


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    es.lib()          # raises LibraryMissing when the CUDA library is absent
    oracle.build()
    yield
    es.set_path_override("auto")


MAXPLUS_DISTS = dict(x_dist=("uniform", -1.0, 1.0), a_dist=("uniform", 0.0, 0.1), init_dist=("const", -3.0e38))
NORMCAP_DISTS = dict(x_dist=("normal", 0.0, 0.5), a_dist=("uniform", 0.8, 1.0), init_dist=("normal", 0.0, 0.2))

SMALL = [
    # lanes innermost, TMA pipeline: ragged lane tiles and a ragged last time tile
    ("lane_tma", wl.custom(T_, (3, 50, 200), 1, name="tanh_lane")),
    ("lane_tma", wl.custom(T_, (2, 257, 64), 1, name="tanh_lane_T257")),
    ("lane_tma", wl.custom(M_, (2, 37, 96), 1, name="maxplus_lane", **MAXPLUS_DISTS)),
    ("lane_tma", wl.custom(M_, (5, 64, 1000), 1, name="maxplus_lane_wide", **MAXPLUS_DISTS)),
    ("lane_tma", wl.custom(T_, (300, 40), 0, name="tanh_lane_axis0")),
    # enough lanes for 256-lane tiles: a ragged last lane tile (1000 = 3 x 256 + 232) and trip tile
    ("lane_tma", wl.custom(T_, (40, 70, 1000), 1, name="tanh_lane_256")),
    ("lane_tma", wl.custom(M_, (40, 70, 1000), 1, name="maxplus_lane_256", **MAXPLUS_DISTS)),
    ("lane_tma", wl.custom(T_, (4, 33, 8, 16), 1, state_axis=True, seq_widths=(16, 16), name="tanh_vec_full")),
    # time innermost, transposed through SMEM
    ("time_tma", wl.custom(T_, (300, 100), -1, name="tanh_time")),
    ("time_tma", wl.custom(T_, (64, 32), -1, name="tanh_time_one_tile")),
    ("time_tma", wl.custom(M_, (129, 68), 1, name="maxplus_time", **MAXPLUS_DISTS)),
    ("time_tma", wl.custom(T_, (2, 3, 96), 2, name="tanh_time_rank3")),
    # NORMCAP vector state
    ("vec_tma", wl.custom(N_, (3, 45, 20, 16), 1, True, (16, 1), name="normcap_w16", **NORMCAP_DISTS)),
    ("vec_tma", wl.custom(N_, (2, 40, 24, 16), 1, True, (16, 16), name="normcap_w16_fullgate", **NORMCAP_DISTS)),
    ("vec_tma", wl.custom(N_, (2, 19, 40, 8), 1, True, (8, 1), name="normcap_w8", **NORMCAP_DISTS)),
    ("vec_tma", wl.custom(N_, (2, 21, 64, 4), 1, True, (4, 4), name="normcap_w4", **NORMCAP_DISTS)),
    ("vec_tma", wl.custom(N_, (1, 17, 128, 2), 1, True, (2, 2), name="normcap_w2", **NORMCAP_DISTS)),
    ("vec_tma", wl.custom(N_, (33, 2, 16, 16), 0, True, (16, 1), name="normcap_axis0", **NORMCAP_DISTS)),
    # the generic kernel
    ("generic", wl.WORKLOADS["tanh_decay_small"]),
    ("generic", wl.custom(T_, (5, 7, 3), 0, name="tanh_odd_axis0")),
    ("generic", wl.custom(T_, (5, 7, 3), -2, name="tanh_odd_axis1")),
    ("generic", wl.custom(M_, (5, 7, 3), 2, name="maxplus_odd_axis2", **MAXPLUS_DISTS)),
    ("generic", wl.custom(N_, (3, 30, 7, 5), 1, True, (5, 1), name="normcap_w5", **NORMCAP_DISTS)),
    ("generic", wl.custom(N_, (2, 25, 3, 16), 1, True, (16, 1), name="normcap_few_lanes", **NORMCAP_DISTS)),
    ("generic", wl.custom(N_, (2, 9, 3, 1), 1, True, (1, 1), name="normcap_w1", **NORMCAP_DISTS)),
    ("generic", wl.custom(T_, (4, 11, 6, 3), 1, True, (3, 1), name="tanh_vec_gate", x_dist=("normal", 0.0, 1.0))),
    ("generic", wl.custom(M_, (4, 11, 6, 3), 1, True, (1, 3), name="maxplus_vec_bcast_x", **MAXPLUS_DISTS)),
    ("generic", wl.custom(T_, (17,), 0, name="tanh_rank1")),
    ("generic", wl.custom(T_, (6, 1, 10), 1, name="tanh_T1")),
]


@pytest.mark.parametrize("path,w", SMALL, ids=[w.name for _, w in SMALL])
@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
def test_small_parity(path, w, reverse):
    check_workload(w, reverse, path=path)


@pytest.mark.parametrize("path,w", [s for s in SMALL if s[0] != "generic"],
                         ids=[w.name for p, w in SMALL if p != "generic"])
def test_generic_kernel_agrees_on_tma_shapes(path, w):
    """The generic kernel, forced on shapes a TMA path would take, meets the
    same bar (a second, independent CUDA implementation of every body)."""
    try:
        es.set_path_override("generic")
        check_workload(w, reverse=True)
    finally:
        es.set_path_override("auto")


def test_generic_normcap_is_bit_exact():
    """The generic kernel adds the squares in state order like the oracle, so
    with correctly rounded sqrt and division NORMCAP matches bit for bit."""
    w = wl.custom(N_, (3, 30, 7, 5), 1, True, (5, 1), **NORMCAP_DISTS)
    init, seqs = wl.make_inputs(w)
    got = run_gpu(w, init, seqs, False).cpu().numpy()
    want = run_oracle(w, init, seqs, False)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_misaligned_pointers_take_the_generic_path():
    w = wl.custom(T_, (3, 40, 64), 1)
    init, (x, a) = wl.make_inputs(w)
    dev = "cuda"
    n = x.numel()
    xb = torch.empty(n + 1, device=dev)
    xb[1:].copy_(x.reshape(-1))
    x_mis = xb[1:].view(x.shape)
    assert x_mis.data_ptr() % 16 != 0
    out = es.scan(T_, init.to(dev), [x_mis, a.to(dev)], axis=1)
    es.device_status()
    compare(T_, out.cpu().numpy(), run_oracle(w, init, [x, a], False), "misaligned x")


def test_empty_lanes_launch_nothing():
    x = torch.zeros((3, 5, 0), device="cuda")
    init = torch.zeros((3, 0), device="cuda")
    before = es.launch_count()
    out = es.scan(T_, init, [x, x.clone()], axis=1)
    assert out.shape == (3, 5, 0)
    assert es.launch_count() == before


def test_out_argument_and_chunked_resume():
    """Feeding the final-state slice of one call as the next call's initial
    state continues the recurrence exactly (chunked resume), on the GPU."""
    w = wl.custom(M_, (2, 96, 64), 1, **MAXPLUS_DISTS)
    init, (x, c) = wl.make_inputs(w, "cuda")
    full = es.scan(M_, init, [x, c], axis=1)
    first = torch.empty((2, 40, 64), device="cuda")
    es.scan(M_, init, [x[:, :40].contiguous(), c[:, :40].contiguous()], axis=1, out=first)
    second = es.scan(M_, first[:, -1].contiguous(), [x[:, 40:].contiguous(), c[:, 40:].contiguous()], axis=1)
    es.device_status()
    assert torch.equal(torch.cat([first, second], 1), full)


def test_streams_are_respected():
    w = wl.custom(T_, (4, 64, 256), 1)
    init, seqs = wl.make_inputs(w, "cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        out = es.scan(T_, init, seqs, axis=1)
    torch.cuda.current_stream().wait_stream(s)
    es.device_status(s)
    compare(T_, out.cpu().numpy(), run_oracle(w, init, seqs, False), "side stream")


# ---------------------------------------------------------------------------
# the five measured workloads at full size, as the bench launches them

FULL = ["tanh_decay_small", "tanh_decay_lanes", "normcap_vector", "maxplus_reverse", "tanh_decay_time_inner"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_element_and_properties(name):
    """Every output value of the workload (each direction it names) against
    the oracle run on all host cores on the same seeded inputs: MAXPLUS bit for
    bit, the float bodies within 1e-5 * (1 + |oracle|); then properties that
    hold at any size (tanh range, the norm cap, the max-plus sweep's tight
    bound)."""
    w = wl.WORKLOADS[name]
    init, seqs = wl.make_inputs(w, "cuda")
    init_h = init.cpu().numpy()
    seqs_h = [s.cpu().numpy() for s in seqs]
    for reverse in w.reverse:
        out = es.scan(w.body, init, seqs, axis=w.axis, state_axis=w.state_axis, reverse=reverse)
        es.device_status()
        want = oracle.scan_threads(w.body, init_h, seqs_h, axis=w.axis, state_axis=w.state_axis, reverse=reverse)
        compare_blocks(w.body, out.cpu().numpy(), want, "%s reverse=%s, every element" % (name, reverse))
        del want
        assert bool(torch.isfinite(out).all())
        x, a = seqs
        if w.body == T_:
            assert float(out.abs().max()) <= 1.0                       # tanh range
        elif w.body == N_:
            n = torch.linalg.vector_norm(out.double(), dim=-1)
            assert float(n.max()) <= 1.0 + 1e-6                         # the cap
        else:
            # reverse max-plus: h[t] >= x[t], h[t] >= h[t+1] - c[t], one of them equal
            ax = w.ax
            nxt = torch.cat([out.narrow(ax, 1, w.T - 1), init.unsqueeze(ax)], dim=ax)
            via = nxt - a
            assert bool((out >= x).all()) and bool((out >= via).all())
            assert bool(((out == x) | (out == via)).all())
        del out
        torch.cuda.empty_cache()


def test_full_size_reverse_equals_flip_scan_flip():
    """At the bench's size: a reverse scan equals flipping the sequences,
    scanning forward and flipping back, bit for bit (MAXPLUS)."""
    w = wl.WORKLOADS["maxplus_reverse"]
    init, (x, c) = wl.make_inputs(w, "cuda")
    rev = es.scan(w.body, init, [x, c], axis=1, reverse=True)
    xf, cf = x.flip(1).contiguous(), c.flip(1).contiguous()
    del x, c
    fwd = es.scan(w.body, init, [xf, cf], axis=1)
    es.device_status()
    assert torch.equal(rev, fwd.flip(1))


@pytest.mark.parametrize("path,shape,axis", [
    ("lane_tma", (2, 40, 64), 1),
    ("time_tma", (70, 64), -1),
    ("generic", (3, 9, 5), 1),
], ids=["lane_tma", "time_tma", "generic"])
@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
def test_maxplus_signed_zeros_and_ties_bitwise(path, shape, axis, reverse):
    """MAXPLUS on values drawn from a small set with signed zeros, so ties
    and +0/-0 meetings are frequent: every path matches the oracle's IEEE
    maximum bit for bit."""
    rng = np.random.default_rng(5)
    x = rng.choice(np.array([-1.0, -0.5, -0.0, 0.0, 0.5, 1.0], np.float32), size=shape).astype(np.float32)
    c = rng.choice(np.array([0.0, -0.0, 0.25, 0.5], np.float32), size=shape).astype(np.float32)
    ax = axis % len(shape)
    ishape = shape[:ax] + shape[ax + 1:]
    init = rng.choice(np.array([-0.0, 0.0, -3.0e38, 0.5], np.float32), size=ishape).astype(np.float32)
    p = es.plan(M_, shape, axis, reverse=reverse)
    assert p["path"] == path
    out = es.scan(M_, torch.from_numpy(init).cuda(), [torch.from_numpy(x).cuda(), torch.from_numpy(c).cuda()],
                  axis=axis, reverse=reverse)
    es.device_status()
    want = oracle.scan(M_, init, [x, c], axis=axis, reverse=reverse)
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    # the inputs really exercised both zero signs
    assert (np.signbit(want) & (want == 0)).any() and (~np.signbit(want) & (want == 0)).any()


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
def test_normcap_vector_path_inside_unit_ball_is_exact(reverse):
    """While every state stays inside the unit ball the cap never acts, and the
    vector-state kernel then reproduces the oracle bit for bit (its scale is
    exactly one there)."""
    w = wl.custom(N_, (2, 40, 24, 16), 1, True, (16, 1), x_dist=("normal", 0.0, 0.01),
                  a_dist=("uniform", 0.5, 0.9), init_dist=("normal", 0.0, 0.01))
    init, seqs = wl.make_inputs(w)
    assert es.plan(N_, w.shape, 1, 16, (16, 1), reverse)["path"] == "vec_tma"
    got = run_gpu(w, init, seqs, reverse).cpu().numpy()
    want = run_oracle(w, init, seqs, reverse)
    assert np.linalg.norm(want.astype(np.float64), axis=-1).max() < 1.0
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
