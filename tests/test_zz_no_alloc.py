"""es_matrix_scan_static_f32: the chunked matrix-scan in the library's own
static device scratch -- no workspace argument and no device allocation per
call; results identical to the workspace entry; successive uses on different
streams ordered; a call needing more scratch than the library owns runs lane
by lane."""
import ctypes
import os

import numpy as np
import pytest

from element_scan_recurrences_gb300 import binding as es

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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


@pytest.mark.gpu
def test_static_scratch_no_allocation_and_same_result():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    a, b = _inputs(4, 3000, 8, 8, 1)
    da, db = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    need = es.matrix_scan_workspace(a.shape, b.shape, 1)
    assert 0 < need <= es.STATIC_SCRATCH_BYTES
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    want = es.matrix_scan_ws(da, db, ws, axis=1)
    out = torch.empty_like(want)
    es.matrix_scan_static(da, db, axis=1, out=out)          # first use loads the module and its scratch
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    n0 = es.launch_count()
    for _ in range(3):
        es.matrix_scan_static(da, db, axis=1, out=out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "a static-scratch call allocated device memory"
    assert es.launch_count() - n0 == 9                      # the chunked scan: three kernels a call
    es.device_status()
    assert torch.equal(out, want)


@pytest.mark.gpu
def test_static_scratch_ordered_across_streams_and_fallback():
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
    for got, (a, b) in ((o1, (a1, b1)), (o2, (a2, b2))):
        want = M.matrix_scan(a, b, axis=1).astype(np.float64)
        err = np.abs(got.cpu().numpy() - want) / (1 + np.abs(want))
        assert err.max() <= 1e-5
    # more scratch than the library owns (one lane of 1024 columns over 65536
    # trips): lane by lane, exactly as es_matrix_scan_f32
    lanes, T, n, m = 1, 65536, 4, 1024
    assert es.matrix_scan_workspace([lanes, T, n, n], [lanes, T, n, m], 1) > es.STATIC_SCRATCH_BYTES
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    a = torch.randn(lanes, T, n, n, generator=g, device="cuda") * 0.2
    b = torch.randn(lanes, T, n, m, generator=g, device="cuda")
    got = es.matrix_scan_static(a, b, axis=1)
    ref = es.matrix_scan(a, b, axis=1)
    es.device_status()
    assert torch.equal(got, ref)
