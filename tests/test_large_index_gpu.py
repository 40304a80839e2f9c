"""Scans past 2**32 elements: every offset into x, a and the states is
64-bit.  One workload each for the lanes-innermost kernel (the headline
path), the time-innermost kernel and a body program's lanes-innermost
kernel, about 17 GB per tensor; lanes at the far end of the buffers (and
the first ones) are checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from element_scan_recurrences_gb300 import binding as es
from oracle.body import scan_body

pytestmark = pytest.mark.gpu

BIG = 1 << 32


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    free, _ = torch.cuda.mem_get_info()
    if free < 64 << 30:
        pytest.skip("needs 64 GB of free device memory")
    es.lib()


def _inputs(shape, gen):
    x = torch.randn(shape, device="cuda", generator=gen)
    a = torch.rand(shape, device="cuda", generator=gen).mul_(0.49).add_(0.5)   # in place: no temporaries
    return x, a


def _close(got, want, what):
    err = np.abs(got.astype(np.float64) - want) / (1.0 + np.abs(want.astype(np.float64)))
    assert float(err.max()) <= 1e-5, "%s: %g" % (what, float(err.max()))


def test_lanes_innermost_past_2_32():
    shape = (2, 512, (1 << 22) + 96)
    assert np.prod(shape) > BIG
    gen = torch.Generator("cuda").manual_seed(0)
    x, a = _inputs(shape, gen)
    init = torch.zeros(shape[0], shape[2], device="cuda")
    assert es.plan(es.TANH_DECAY, shape, 1)["path"] == "lane_tma"
    out = es.scan(es.TANH_DECAY, init, [x, a], axis=1)
    es.device_status()
    for o, lanes in ((0, [0, 1]), (1, [shape[2] - 1, shape[2] - 97, shape[2] // 2])):
        xs, as_ = x[o, :, lanes].cpu().numpy(), a[o, :, lanes].cpu().numpy()
        want = oracle.scan(es.TANH_DECAY, np.zeros((len(lanes),), np.float32), [xs, as_], axis=0)
        _close(out[o, :, lanes].cpu().numpy(), want, "lanes o=%d" % o)
    del x, a, out, init
    torch.cuda.empty_cache()


def test_time_innermost_past_2_32():
    shape = ((1 << 22) + 1, 1024)
    assert np.prod(shape) > BIG
    gen = torch.Generator("cuda").manual_seed(1)
    x, a = _inputs(shape, gen)
    init = torch.zeros(shape[0], device="cuda")
    for reverse in (False, True):
        assert es.plan(es.TANH_DECAY, shape, -1, reverse=reverse)["path"] == "time_tma"
        out = es.scan(es.TANH_DECAY, init, [x, a], axis=-1, reverse=reverse)
        es.device_status()
        rows = [0, shape[0] - 1, shape[0] - 2]
        want = oracle.scan(es.TANH_DECAY, np.zeros(len(rows), np.float32),
                           [x[rows].cpu().numpy(), a[rows].cpu().numpy()], axis=-1, reverse=reverse)
        _close(out[rows].cpu().numpy(), want, "rows reverse=%s" % reverse)
        del out
    del x, a, init
    torch.cuda.empty_cache()


def test_body_program_past_2_32():
    text = "(lambda (h x a) (+ (* a h) x))"        # IEEE-exact: bit for bit
    shape = (2, 512, (1 << 22) + 96)
    gen = torch.Generator("cuda").manual_seed(2)
    x, a = _inputs(shape, gen)
    init = torch.zeros(shape[0], shape[2], device="cuda")
    body = es.Body(text)
    assert body.plan(list(shape), 1)["path"] == "lane_tma"
    out = body.scan(init, [x, a], axis=1)
    es.device_status()
    lanes = [shape[2] - 1, shape[2] - 33, 5]
    want = scan_body(text, np.zeros((1, len(lanes)), np.float32),
                     [x[1:2, :, lanes].cpu().numpy(), a[1:2, :, lanes].cpu().numpy()], axis=1)
    assert np.array_equal(out[1:2, :, lanes].cpu().numpy(), want)
    del x, a, out, init
    torch.cuda.empty_cache()
