"""matrix-scan and linear-scan through the C ABI without a GPU: the library
rejects the shapes the oracle rejects and plans the documented kernels."""
import numpy as np
import pytest

import matrix_pins
import oracle.matrix as M
from element_scan_recurrences_gb300 import binding as es


@pytest.mark.parametrize("case", matrix_pins.REJECTED, ids=[str(r) for r in matrix_pins.REJECTED])
def test_library_rejects_what_the_oracle_rejects(case):
    sa, sb, axis = case
    with pytest.raises(ValueError):
        M.matrix_scan(np.zeros(sa, np.float32), np.zeros(sb, np.float32), axis=axis)
    with pytest.raises(es.EsError) as e:
        es.plan_matrix_scan(sa, sb, axis)
    assert e.value.status == 1


def test_matrix_plans():
    p = es.plan_matrix_scan([64, 1024, 16, 16, 16], [64, 1024, 16, 16, 16], axis=1)
    assert p["path"] == "mat_tma" and (p["O"], p["T"], p["J"], p["W"]) == (64, 1024, 16, 256)
    # broadcast a (shared by the batch), odd n, or n*m not a multiple of 4: generic
    assert es.plan_matrix_scan([1, 1024, 1, 16, 16], [64, 1024, 16, 16, 16], axis=1)["path"] == "generic"
    assert es.plan_matrix_scan([8, 100, 3, 3], [8, 100, 3, 5], axis=1)["path"] == "generic"
    assert es.plan_matrix_scan([8, 100, 2, 2], [8, 100, 2, 1], axis=1)["path"] == "generic"
    assert es.plan_matrix_scan([8, 100, 2, 2], [8, 100, 2, 2], axis=1)["path"] == "mat_tma"
    # projective: n + m <= 32
    assert es.plan_matrix_scan([8, 100, 16, 16], [8, 100, 16, 16], axis=1, projective=True)["path"] == "mat_tma"
    with pytest.raises(es.EsError) as e:
        es.plan_matrix_scan([8, 100, 16, 16], [8, 100, 16, 17], axis=1, projective=True)
    assert e.value.status == 4
    # empty lanes
    assert es.plan_matrix_scan([0, 100, 4, 4], [0, 100, 4, 4], axis=1)["path"] == "empty"
    # the axis counts among the leading dims
    p = es.plan_matrix_scan([5, 7, 4, 4], [5, 7, 4, 3], axis=-1)
    assert (p["O"], p["T"], p["J"]) == (5, 7, 1)
    # out may not overlap an input
    with pytest.raises(es.EsError) as e:
        es.plan_matrix_scan([5, 7, 4, 4], [5, 7, 4, 4], axis=0, ptrs=[1 << 44, 2 << 44, (1 << 44) + 16])
    assert e.value.status == 3


def test_linear_plans():
    assert es.plan_linear_scan([64, 4096, 1024], [64, 4096, 1024], axis=1)["path"] == "lane_tma"
    assert es.plan_linear_scan([262144, 1024], [262144, 1024], axis=-1)["path"] == "time_tma"
    assert es.plan_linear_scan([], [64, 4096, 1024], axis=1)["path"] == "generic"        # a number
    assert es.plan_linear_scan([64, 1, 1024], [64, 4096, 1024], axis=1)["path"] == "generic"
    with pytest.raises(es.EsError):
        es.plan_linear_scan([3, 4], [4, 4], axis=0)


def test_workspace_plans():
    """Few long lanes with a workspace: the chunked scan on the TMA passes
    where they take the operands, else on the direct-load chunk kernels;
    without enough workspace the sequential path; forcing checked."""
    sa, sb = [8, 131072, 16, 16], [8, 131072, 16, 16]
    need = es.matrix_scan_workspace(sa, sb, 1)
    # 8 lanes x 38 CTAs of 4 chunks: one wave of 152 SMs x 2 CTAs, so 152
    # chunks of 863 trips per lane
    assert need == 8 * 152 * (16 * 16 + 2 * 16 * 16) * 4
    assert es.plan_matrix_scan_ws(sa, sb, need, axis=1)["path"] == "mat_chunked_tma"
    assert es.plan_matrix_scan_ws(sa, sb, need, axis=1, reverse=True)["path"] == "mat_chunked_tma"
    assert es.plan_matrix_scan_ws(sa, sb, need - 16, axis=1)["path"] == "mat_tma"
    assert es.plan_matrix_scan_ws(sa, sb, 0, axis=1)["path"] == "mat_tma"
    # odd n, n + m > 32, n*m not a multiple of 4, a broadcast a: direct-load chunk kernels
    for a_shape, b_shape in (([3, 2000, 7, 7], [3, 2000, 7, 2]), ([3, 2000, 16, 16], [3, 2000, 16, 17]),
                             ([3, 2000, 2, 2], [3, 2000, 2, 1]), ([1, 2000, 4, 4], [3, 2000, 4, 4])):
        n = es.matrix_scan_workspace(a_shape, b_shape, 1)
        assert n > 0
        assert es.plan_matrix_scan_ws(a_shape, b_shape, n, axis=1)["path"] == "mat_chunked", (a_shape, b_shape)
    # an `out` off the 16-byte grid takes the direct-load kernels too
    p = es.plan_matrix_scan_ws(sa, sb, need, axis=1, ptrs=[1 << 44, 2 << 44, (3 << 44) + 4, 4 << 44])
    assert p["path"] == "mat_chunked"
    # many lanes: no chunking
    assert es.matrix_scan_workspace([64, 1024, 16, 16, 16], [64, 1024, 16, 16, 16], 1) == 0
    assert es.plan_matrix_scan_ws([64, 1024, 16, 16, 16], [64, 1024, 16, 16, 16], 1 << 20, axis=1)["path"] == "mat_tma"
    # forcing
    es.set_path_override("mat_chunked")
    try:
        assert es.plan_matrix_scan_ws(sa, sb, need, axis=1)["path"] == "mat_chunked"
        with pytest.raises(es.EsError) as e:
            es.plan_matrix_scan_ws(sa, sb, need - 16, axis=1)
        assert e.value.status == 4
    finally:
        es.set_path_override("auto")
    es.set_path_override("mat_chunked_tma")
    try:
        assert es.plan_matrix_scan_ws(sa, sb, need, axis=1)["path"] == "mat_chunked_tma"
        n = es.matrix_scan_workspace([3, 2000, 7, 7], [3, 2000, 7, 2], 1)
        with pytest.raises(es.EsError) as e:
            es.plan_matrix_scan_ws([3, 2000, 7, 7], [3, 2000, 7, 2], n, axis=1)
        assert e.value.status == 4
    finally:
        es.set_path_override("auto")
    # the workspace may not overlap an operand, and sits on the 16-byte grid
    with pytest.raises(es.EsError) as e:
        es.plan_matrix_scan_ws(sa, sb, need, axis=1, ptrs=[1 << 44, 2 << 44, 3 << 44, (1 << 44) + 64])
    assert e.value.status == 3
    with pytest.raises(es.EsError) as e:
        es.plan_matrix_scan_ws(sa, sb, need, axis=1, ptrs=[1 << 44, 2 << 44, 3 << 44, (4 << 44) + 4])
    assert e.value.status == 3


def test_backward_workspace_plans():
    """The gradient with a workspace: the cotangent scan chunked on the TMA
    passes where the forward would be, with the forward's workspace size;
    else the sequential gradient; forcing checked."""
    sa, sb = [8, 131072, 16, 16], [8, 131072, 16, 16]
    need = es.matrix_scan_workspace(sa, sb, 1)
    for reverse in (False, True):
        p = es.plan_matrix_scan_backward_ws(sa, sb, need, axis=1, reverse=reverse)
        assert p["path"] == "mat_chunked_tma" and p["reverse"] == reverse
    assert es.plan_matrix_scan_backward_ws(sa, sb, need - 16, axis=1)["path"] == "mat_tma"
    assert es.plan_matrix_scan_backward_ws(sa, sb, 0, axis=1)["path"] == "mat_tma"
    # operands the TMA passes do not take: the sequential gradient
    n = es.matrix_scan_workspace([3, 2000, 7, 7], [3, 2000, 7, 2], 1)
    assert es.plan_matrix_scan_backward_ws([3, 2000, 7, 7], [3, 2000, 7, 2], n, axis=1)["path"] == "generic"
    # a projective scan has no gradient
    with pytest.raises(es.EsError) as e:
        es.plan_matrix_scan_backward_ws(sa, sb, need, axis=1, projective=True)
    assert e.value.status == 3
    # the workspace may not overlap an operand (here grad_b)
    with pytest.raises(es.EsError) as e:
        es.plan_matrix_scan_backward_ws(sa, sb, need, axis=1, ptrs=[(k + 1) << 44 for k in range(6)] + [(6 << 44) + 64])
    assert e.value.status == 3
    es.set_path_override("mat_chunked_tma")
    try:
        assert es.plan_matrix_scan_backward_ws(sa, sb, need, axis=1)["path"] == "mat_chunked_tma"
        for args in ((sa, sb, need - 16), ([3, 2000, 7, 7], [3, 2000, 7, 2], n)):
            with pytest.raises(es.EsError) as e:
                es.plan_matrix_scan_backward_ws(*args, axis=1)
            assert e.value.status == 4
        # the entry without a workspace cannot take it
        with pytest.raises(es.EsError) as e:
            es.plan_matrix_scan_backward(sa, sb, axis=1)
        assert e.value.status == 4
    finally:
        es.set_path_override("auto")
    es.set_path_override("mat_chunked")   # the direct-load chunk kernels have no gradient
    try:
        with pytest.raises(es.EsError) as e:
            es.plan_matrix_scan_backward_ws(sa, sb, need, axis=1)
        assert e.value.status == 4
    finally:
        es.set_path_override("auto")


@pytest.mark.parametrize("n,m,lead,T,chunks", [
    # TMA passes: lanes * ceil(chunks / LPC) CTAs fill one wave of 152 SMs x 2
    (16, 16, (8,), 131072, 152),        # LPC 4: 38 CTAs a lane
    (16, 16, (400,), 100000, 4),        # more lanes than a wave's CTAs: one CTA a lane
    (4, 4, (2,), 100000, 607),          # LPC 4: 152 CTAs a lane, 608 asked; chunks of 165 trips need 607
    (16, 16, (3,), 3001, 46),           # capped at chunks of 64 trips
    # direct-load kernels (n = 7): about 4096 (lane, chunk) units, capped the same way
    (7, 2, (3,), 2000, 31),
    (7, 2, (1,), 1 << 20, 4096),
])
def test_chunk_count(n, m, lead, T, chunks):
    """The chunk count behind es_matrix_scan_workspace_f32 (host logic): the
    workspace is lanes x chunks units of n*n + 2*n*m floats."""
    a_shape = [lead[0], T] + list(lead[1:]) + [n, n]
    b_shape = [lead[0], T] + list(lead[1:]) + [n, m]
    lanes = int(np.prod(lead))
    assert es.matrix_scan_workspace(a_shape, b_shape, 1) == lanes * chunks * (n * n + 2 * n * m) * 4
