"""table-scan through the C ABI without a GPU: plans and rejections."""
import pytest

from element_scan_recurrences_gb300 import binding as es


def test_table_plans():
    assert es.plan_table_scan(64, 16, [262144, 1024])["path"] == "time_tma"
    assert es.plan_table_scan(64, 16, [64, 4096, 1024], axis=1)["path"] == "lane_tma"
    assert es.plan_table_scan(64, 16, [64, 4096, 30], axis=1)["path"] == "generic"
    assert es.plan_table_scan(64, 16, [5, 30])["path"] == "generic"            # T not a multiple of 4
    assert es.plan_table_scan(2, 2, [5, 0])["path"] == "empty"                  # an empty axis
    p = es.plan_table_scan(3, 4, [2, 7, 5], axis=1)
    assert (p["O"], p["T"], p["J"]) == (2, 7, 5)


@pytest.mark.parametrize("args", [
    (0, 2, [3, 4], -1, 0),        # no states
    (2, 0, [3, 4], -1, 0),        # no symbols
    (2, 2, [3, 4], 2, 0),         # axis out of range
    (2, 2, [3, 4], -3, 0),        # axis out of range
    (2, 2, [3, 4], -1, 2),        # start not a state
    (2, 2, [3, 4], -1, -1),       # start not a state
])
def test_table_rejections(args):
    n_states, n_syms, shape, axis, start = args
    with pytest.raises(es.EsError) as e:
        es.plan_table_scan(n_states, n_syms, shape, axis=axis, start=start)
    assert e.value.status == 1


def test_table_overlap_and_size():
    with pytest.raises(es.EsError) as e:
        es.plan_table_scan(2, 2, [3, 4], ptrs=[1 << 44, 2 << 44, (2 << 44) + 8])
    assert e.value.status == 3
    with pytest.raises(es.EsError) as e:
        es.plan_table_scan(1 << 16, 1 << 16, [3, 4])
    assert e.value.status == 4
