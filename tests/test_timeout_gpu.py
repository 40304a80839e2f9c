"""Bounded device waits: when a pipeline tile never arrives, the kernel gives
up after the wait limit, records ES_E_TIMEOUT in the device status word and
returns; the context stays usable and the next call is correct.

The missing tile is made on the host side of the pipeline (the producer is
told to skip one load), never by faulting or hanging the GPU.
"""
import pytest
import torch

from element_scan_recurrences_gb300 import binding as es
from element_scan_recurrences_gb300 import workloads as wl
from parity_helpers import compare, run_oracle

pytestmark = pytest.mark.gpu

CASES = [
    ("lane_tma", wl.custom(wl.TANH_DECAY, (2, 400, 64), 1, name="lane")),
    ("time_tma", wl.custom(wl.MAXPLUS, (130, 400), -1, name="time", x_dist=("uniform", -1.0, 1.0),
                           a_dist=("uniform", 0.0, 0.1), init_dist=("const", -3.0e38))),
    ("vec_tma", wl.custom(wl.NORMCAP, (2, 400, 16, 16), 1, True, (16, 1), name="vec",
                          x_dist=("normal", 0.0, 0.5), a_dist=("uniform", 0.8, 1.0))),
]


@pytest.fixture(autouse=True)
def restore():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    es.set_drop_tile(-1)
    es.set_wait_limit_ns(2_000_000_000)
    es.set_path_override("auto")


@pytest.mark.parametrize("path,w", CASES, ids=[c[0] for c in CASES])
def test_dropped_tile_times_out_then_recovers(path, w):
    init, seqs = wl.make_inputs(w, "cuda")
    reverse = w.reverse[0]
    es.set_path_override(path)
    es.device_status()                    # clean status word
    es.set_wait_limit_ns(20_000_000)      # 20 ms
    es.set_drop_tile(3)
    es.scan(w.body, init, seqs, axis=w.axis, state_axis=w.state_axis, reverse=reverse)
    with pytest.raises(es.EsError) as ei:
        es.device_status()
    assert ei.value.status == 6           # ES_E_TIMEOUT
    es.device_status()                    # the word was cleared
    es.set_drop_tile(-1)
    es.set_wait_limit_ns(2_000_000_000)
    out = es.scan(w.body, init, seqs, axis=w.axis, state_axis=w.state_axis, reverse=reverse)
    es.device_status()
    compare(w.body, out.cpu().numpy(), run_oracle(w, init, seqs, reverse), "after recovery " + path)


def test_backward_dropped_tile_times_out_then_recovers():
    w = wl.custom(wl.TANH_DECAY, (2, 400, 64), 1, name="bwd")
    init, seqs = wl.make_inputs(w, "cuda")
    states = es.scan(w.body, init, seqs, axis=1)
    G = torch.ones_like(states)
    assert es.plan_backward(w.body, w.shape, 1)["path"] == "lane_tma"
    es.device_status()
    es.set_wait_limit_ns(20_000_000)
    es.set_drop_tile(2)
    es.scan_backward(w.body, init, seqs, states, G, axis=1)
    with pytest.raises(es.EsError) as ei:
        es.device_status()
    assert ei.value.status == 6
    es.set_drop_tile(-1)
    es.set_wait_limit_ns(2_000_000_000)
    gi, gs = es.scan_backward(w.body, init, seqs, states, G, axis=1)
    es.device_status()
    try:
        es.set_path_override("generic")
        gi2, gs2 = es.scan_backward(w.body, init, seqs, states, G, axis=1)
        es.device_status()
    finally:
        es.set_path_override("auto")
    assert torch.equal(gi, gi2) and torch.equal(gs[0], gs2[0]) and torch.equal(gs[1], gs2[1])
