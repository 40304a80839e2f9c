"""End-to-end calls on host buffers (es_scan_host_f32, es_scan_body_host_f32):
the row pieces pipelined over the library's copy and compute streams give
the bits of one device scan of the whole call, and the call stays ordered
with the caller's stream."""
import numpy as np
import pytest
import torch

import body_cases
from element_scan_recurrences_gb300 import binding as es
from element_scan_recurrences_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    es.lib()


def _host(w, pinned=True):
    init, seqs = wl.make_inputs(w, "cpu")
    f = (lambda t: t.contiguous().pin_memory()) if pinned else (lambda t: t.contiguous())
    return f(init), [f(s) for s in seqs]


def _device_like(init_h, seqs_h, shape):
    return (torch.empty(init_h.shape, device="cuda"), [torch.empty(s.shape, device="cuda") for s in seqs_h],
            torch.empty(shape, device="cuda"))


@pytest.mark.parametrize("chunks", [0, 1, 3, 13, 64])
@pytest.mark.parametrize("reverse", [False, True])
def test_fixed_body_pieces_match_one_scan(chunks, reverse):
    w = wl.custom(wl.TANH_DECAY, (13, 57, 40), 1)
    init_h, seqs_h = _host(w)
    want = es.scan(w.body, init_h.cuda(), [s.cuda() for s in seqs_h], axis=1, reverse=reverse).cpu()
    out_h = torch.empty(w.shape).pin_memory()
    es.scan_host(w.body, init_h, seqs_h, out_h, _device_like(init_h, seqs_h, w.shape), axis=1, reverse=reverse,
                 chunks=chunks)
    torch.cuda.current_stream().synchronize()
    es.device_status()
    assert torch.equal(out_h, want)


def test_axis_first_runs_whole_and_state_axis():
    w = wl.custom(wl.MAXPLUS, (40, 6, 24), 0, x_dist=("uniform", -1.0, 1.0), a_dist=("uniform", 0.0, 0.1))
    init_h, seqs_h = _host(w)
    want = es.scan(w.body, init_h.cuda(), [s.cuda() for s in seqs_h], axis=0).cpu()
    out_h = torch.empty(w.shape).pin_memory()
    es.scan_host(w.body, init_h, seqs_h, out_h, _device_like(init_h, seqs_h, w.shape), axis=0, chunks=8)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(out_h, want)
    v = wl.custom(wl.NORMCAP, (5, 30, 8, 16), 1, True, (16, 1), x_dist=("normal", 0.0, 0.5),
                  a_dist=("uniform", 0.8, 1.0), init_dist=("const", 0.0))
    init_h, seqs_h = _host(v, pinned=False)          # page-able host memory works too
    want = es.scan(v.body, init_h.cuda(), [s.cuda() for s in seqs_h], axis=1, state_axis=True).cpu()
    out_h = torch.empty(v.shape)
    es.scan_host(v.body, init_h, seqs_h, out_h, _device_like(init_h, seqs_h, v.shape), axis=1, state_axis=True,
                 chunks=4)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(out_h, want)


def test_body_program_pieces():
    c = body_cases.case("gated_tanh")
    initial, seqs, _ = body_cases.make_inputs(c, 9, 33, 40, seed=2)
    body = es.Body(c[1])
    want = body.scan(torch.from_numpy(initial).cuda(), [torch.from_numpy(s).cuda() for s in seqs], axis=1).cpu()
    init_h = torch.from_numpy(initial).pin_memory()
    seqs_h = [torch.from_numpy(s).pin_memory() for s in seqs]
    out_h = torch.empty(want.shape).pin_memory()
    body.scan_host(init_h, seqs_h, out_h, _device_like(init_h, seqs_h, want.shape), axis=1, chunks=4)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(out_h, want)


def test_ordering_with_the_callers_stream():
    """Two calls into the same device and host buffers on a side stream,
    then work on that stream reading the device output: every step waits for
    the one before it."""
    w = wl.custom(wl.TANH_DECAY, (16, 40, 64), 1)
    init_h, seqs_h = _host(w)
    init2 = (init_h * 0.5).pin_memory()
    want1 = es.scan(w.body, init_h.cuda(), [s.cuda() for s in seqs_h], axis=1).cpu()
    want2 = es.scan(w.body, init2.cuda(), [s.cuda() for s in seqs_h], axis=1).cpu()
    bufs = _device_like(init_h, seqs_h, w.shape)
    out1 = torch.empty(w.shape).pin_memory()
    out2 = torch.empty(w.shape).pin_memory()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        es.scan_host(w.body, init_h, seqs_h, out1, bufs, axis=1, stream=s, chunks=5)
        es.scan_host(w.body, init2, seqs_h, out2, bufs, axis=1, stream=s, chunks=5)
        after = bufs[2].clone()
    s.synchronize()
    assert torch.equal(out1, want1) and torch.equal(out2, want2)
    assert torch.equal(after.cpu(), want2)


def test_refusals():
    w = wl.custom(wl.TANH_DECAY, (4, 10, 8), 1)
    init_h, seqs_h = _host(w)
    bufs = _device_like(init_h, seqs_h, w.shape)
    with pytest.raises(TypeError):        # a device tensor where host memory is expected
        es.scan_host(w.body, init_h.cuda(), seqs_h, torch.empty(w.shape), bufs, axis=1)
    with pytest.raises(es.EsError) as e:
        es.scan_host(w.body, init_h, seqs_h, torch.empty(w.shape), bufs, axis=1, chunks=65)
    assert e.value.status == 3
