"""es_matrix_scan_static_f32: the chunked matrix-scan (few long lanes) for
callers that cannot allocate device memory -- code where cudaMalloc is
unavailable or not allowed, such as a host application that owns every
allocation.  Its scratch is a static device array the library holds, so a call
allocates nothing and takes no workspace; its results must equal the
workspace entry's on the same inputs, on consecutive calls that reuse the
array; a scan that would need more scratch than the array holds is refused.

This file is collected last, so that a run stopping at the first failure has
run every other test; it passes alone in a fresh process as well."""
import os

import numpy as np
import pytest

from element_scan_recurrences_gb300 import binding as es

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
RTOL = 1e-5


def test_static_entry_is_declared_and_exported():
    header = open(os.path.join(ROOT, "include", "es.h")).read()
    assert "es_matrix_scan_static_f32(" in header and "ES_STATIC_SCRATCH_BYTES" in header
    assert hasattr(es.lib(), "es_matrix_scan_static_f32")
    assert "es_matrix_scan_static_f32" in es.EXPORTS


def _inputs(lanes, T, n, m, seed):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((lanes, T, n, n))
    a = (a / np.linalg.norm(a, ord=2, axis=(-2, -1))[..., None, None] * 0.97).astype(np.float32)
    b = rng.standard_normal((lanes, T, n, m)).astype(np.float32)
    return a, b


def _close(got, want, what):
    got = got.double().cpu().numpy()
    want = want.double().cpu().numpy()
    err = np.abs(got - want) / (1.0 + np.abs(want))
    assert float(err.max()) <= RTOL, "%s: max scaled error %.3g" % (what, float(err.max()))


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_on_consecutive_calls():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    a, b = _inputs(4, 3000, 8, 8, 1)
    da, db = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    need = es.matrix_scan_workspace(a.shape, b.shape, 1)
    assert 0 < need <= es.STATIC_SCRATCH_BYTES
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    want = es.matrix_scan_ws(da, db, ws, axis=1)
    # a second problem, so the second call runs over the first one's scratch values
    a2, b2 = _inputs(3, 2500, 8, 4, 2)
    da2, db2 = torch.from_numpy(a2).cuda(), torch.from_numpy(b2).cuda()
    ws2 = torch.empty(es.matrix_scan_workspace(a2.shape, b2.shape, 1), dtype=torch.uint8, device="cuda")
    want2 = es.matrix_scan_ws(da2, db2, ws2, axis=1)
    for sa, sb, nb in ((a.shape, b.shape, need), (a2.shape, b2.shape, ws2.numel())):
        assert nb <= es.STATIC_SCRATCH_BYTES
        assert es.plan_matrix_scan_ws(sa, sb, nb, axis=1)["path"] in ("mat_chunked_tma", "mat_chunked")
    out, out2 = torch.empty_like(want), torch.empty_like(want2)
    # the first call on the device is the set-up: it loads the library's
    # module, which brings the static array into device memory, and fetches
    # its address; the calls after it allocate nothing
    es.matrix_scan_static(da2, db2, axis=1, out=out2)
    out2.fill_(float("nan"))
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    n0 = es.launch_count()
    es.matrix_scan_static(da, db, axis=1, out=out)        # two calls in a row over the same array
    es.matrix_scan_static(da2, db2, axis=1, out=out2)
    torch.cuda.synchronize()
    es.device_status()
    assert torch.cuda.mem_get_info()[0] == free0, "a static-scratch call allocated device memory"
    assert es.launch_count() - n0 == 6                    # the chunked scan: three kernels a call
    _close(out, want, "first call")
    _close(out2, want2, "second call")
    assert torch.equal(out, want) and torch.equal(out2, want2)   # the same kernels, the same bits


@pytest.mark.gpu
def test_static_scratch_ordered_across_streams():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle.matrix as M
    a1, b1 = _inputs(3, 2000, 4, 4, 2)
    a2, b2 = _inputs(3, 2500, 4, 4, 3)
    d = [torch.from_numpy(t).cuda() for t in (a1, b1, a2, b2)]
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s1):
        o1 = es.matrix_scan_static(d[0], d[1], axis=1, stream=s1)
    with torch.cuda.stream(s2):
        o2 = es.matrix_scan_static(d[2], d[3], axis=1, stream=s2)
    torch.cuda.synchronize()
    es.device_status()
    for got, (a, b) in ((o1, (a1, b1)), (o2, (a2, b2))):
        want = M.matrix_scan(a, b, axis=1).astype(np.float64)
        err = np.abs(got.cpu().numpy() - want) / (1 + np.abs(want))
        assert err.max() <= RTOL


@pytest.mark.gpu
def test_static_scratch_refuses_scans_larger_than_the_array():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    # one lane of 1024 columns over 65536 trips: more scratch than the library holds
    lanes, T, n, m = 1, 65536, 4, 1024
    assert es.matrix_scan_workspace([lanes, T, n, n], [lanes, T, n, m], 1) > es.STATIC_SCRATCH_BYTES
    a = torch.zeros(lanes, T, n, n, device="cuda")
    b = torch.zeros(lanes, T, n, m, device="cuda")
    out = torch.empty_like(b)
    n0 = es.launch_count()
    with pytest.raises(es.EsError) as e:
        es.matrix_scan_static(a, b, axis=1, out=out)
    assert e.value.status == 4 and "ES_STATIC_SCRATCH_BYTES" in e.value.message
    assert es.launch_count() == n0
