"""The C-ABI library on the CPU: it loads, exports every function the header
declares, and its host logic (validation, canonical view, path choice) behaves
as the header documents.  No kernel is launched here."""
import os
import re

import pytest

import element_scan_recurrences_gb300 as es
from element_scan_recurrences_gb300 import binding, workloads

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "es.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    from element_scan_recurrences_gb300 import build
    build.build()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(es_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_binding_exports():
    assert declared_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol():
    L = binding.lib()
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings():
    for code, name in binding.STATUS.items():
        assert es.status_string(code) == name


def test_launch_count_starts_at_zero_without_launches():
    assert es.launch_count() == 0


@pytest.mark.parametrize("name,path", [
    ("tanh_decay_small", "generic"),
    ("tanh_decay_lanes", "lane_tma"),
    ("normcap_vector", "vec_tma"),
    ("maxplus_reverse", "lane_tma"),
    ("tanh_decay_time_inner", "time_tma"),
])
def test_plan_of_each_workload(name, path):
    w = workloads.WORKLOADS[name]
    p = es.plan(w.body, w.shape, w.axis, w.shape[-1] if w.state_axis else 0,
                w.seq_widths if w.state_axis else None, w.reverse[0])
    assert p["path"] == path
    assert p["elements"] == w.elements
    assert p["T"] == w.T
    if name == "normcap_vector":
        assert (p["O"], p["J"], p["W"], p["seq_width"]) == (32, 64, 16, (16, 1))
    if name == "tanh_decay_time_inner":
        assert (p["O"], p["J"], p["W"]) == (262144, 1, 1)


def _err(fn):
    with pytest.raises(es.EsError) as ei:
        fn()
    return ei.value.status, ei.value.message


def test_errors_follow_the_error_table():
    T, N, M = es.TANH_DECAY, es.NORMCAP, es.MAXPLUS
    assert _err(lambda: es.plan(7, [2, 3], 0))[0] == 3                       # unknown body
    st, msg = _err(lambda: es.plan(T, [2, 3, 4], 3))                         # axis out of range
    assert st == 1 and "E-DIM-001" in msg and "[2, 3, 4]" in msg
    assert _err(lambda: es.plan(T, [2, 3, 4], -4))[0] == 1
    assert _err(lambda: es.plan(T, [2, 0, 4], 1))[0] == 1                    # empty sequence axis
    assert _err(lambda: es.plan(T, [2, -1, 4], 1))[0] == 1                   # negative dim
    assert _err(lambda: es.plan(N, [2, 3, 4], 1))[0] == 4                    # NORMCAP needs a state axis
    assert _err(lambda: es.plan(N, [2, 3, 4], -1, 4))[0] == 1                # state axis == sequence axis
    assert _err(lambda: es.plan(N, [2, 3, 17], 1, 17))[0] == 1               # more than 16 values
    assert _err(lambda: es.plan(N, [2, 3, 4], 1, 5))[0] == 1                 # width != last dim
    st, msg = _err(lambda: es.plan(N, [2, 3, 4], 1, 4, (4, 3)))              # gate width not 1 or W
    assert st == 1 and "[2, 3, 3]" in msg
    assert _err(lambda: es.plan(M, [2, 3, 4], 1, 0, (4, 3)))[0] == 1         # scalar state: full widths only
    assert _err(lambda: es.plan(T, [1] * 9, 0))[0] == 4                       # rank above the maximum


def test_pointer_rules():
    base = 1 << 40
    # out overlapping x
    st, msg = _err(lambda: es.plan(es.TANH_DECAY, [4, 8], 0, ptrs=[base, base + 4096, base + 8192, base + 4100]))
    assert st == 3 and "overlaps" in msg
    # misaligned pointer
    assert _err(lambda: es.plan(es.TANH_DECAY, [4, 8], 0, ptrs=[base + 2, 2 * base, 3 * base, 4 * base]))[0] == 3
    # null pointer with work to do
    assert _err(lambda: es.plan(es.TANH_DECAY, [4, 8], 0, ptrs=[0, 2 * base, 3 * base, 4 * base]))[0] == 3
    # 4-byte but not 16-byte aligned data falls back to the generic kernel
    p = es.plan(es.TANH_DECAY, [4, 64, 128], 1, ptrs=[base, 2 * base + 4, 3 * base, 4 * base])
    assert p["path"] == "generic"


def test_empty_lanes_plan_nothing():
    p = es.plan(es.TANH_DECAY, [0, 5, 3], 1, ptrs=[0, 0, 0, 0])
    assert p["path"] == "empty" and p["elements"] == 0
    p = es.plan(es.NORMCAP, [3, 5, 0, 16], 1, 16, (16, 1), ptrs=[0, 0, 0, 0])
    assert p["path"] == "empty"


def test_path_choice_rules():
    P = lambda *a, **k: es.plan(*a, **k)["path"]
    assert P(es.TANH_DECAY, [8, 100, 64], 1) == "lane_tma"
    assert P(es.TANH_DECAY, [8, 100, 30], 1) == "generic"          # row not a multiple of 4 floats
    assert P(es.MAXPLUS, [8, 100, 16], 1) == "generic"              # narrower than one warp of lanes
    assert P(es.TANH_DECAY, [300, 64], -1) == "time_tma"
    assert P(es.TANH_DECAY, [300, 66], -1) == "generic"            # row stride not 16 bytes
    assert P(es.MAXPLUS, [300, 16], 1) == "generic"                # fewer trips than one tile
    assert P(es.NORMCAP, [4, 50, 64, 16], 1, 16, (16, 1)) == "vec_tma"
    assert P(es.NORMCAP, [4, 50, 64, 16], 1, 16, (16, 16)) == "vec_tma"
    assert P(es.NORMCAP, [4, 50, 6, 16], 1, 16, (16, 1)) == "generic"   # fewer lanes than a tile
    assert P(es.NORMCAP, [4, 50, 64, 5], 1, 5, (5, 1)) == "generic"     # width not a power of two
    assert P(es.NORMCAP, [4, 50, 64, 16], 1, 16, (1, 16)) == "generic"  # x broadcast
    assert P(es.TANH_DECAY, [4, 50, 64, 16], 1, 16, (16, 1)) == "generic"
    assert P(es.TANH_DECAY, [4, 50, 64, 16], 1, 16, (16, 16)) == "lane_tma"


def test_path_override_is_checked():
    try:
        es.set_path_override("time_tma")
        assert _err(lambda: es.plan(es.TANH_DECAY, [8, 100, 64], 1))[0] == 4
        es.set_path_override("generic")
        assert es.plan(es.TANH_DECAY, [8, 100, 64], 1)["path"] == "generic"
    finally:
        es.set_path_override("auto")
    assert _err(lambda: es.set_path_override(99))[0] == 3


def test_backward_plans_and_rules():
    T, N, M = es.TANH_DECAY, es.NORMCAP, es.MAXPLUS
    assert es.plan_backward(T, [64, 4096, 1024], 1)["path"] == "lane_tma"
    assert es.plan_backward(M, [128, 16384, 128], 1, reverse=True)["path"] == "lane_tma"
    assert es.plan_backward(N, [32, 8192, 64, 16], 1, 16, (16, 1))["path"] == "vec_tma"
    assert es.plan_backward(N, [3, 30, 7, 16], 1, 16, (16, 1))["path"] == "generic"
    assert es.plan_backward(T, [300, 64], -1)["path"] == "time_tma"
    assert es.plan_backward(T, [300, 36], -1)["path"] == "generic"
    assert es.plan_backward(T, [0, 4, 8], 1, ptrs=[0] * 8)["path"] == "empty"
    base = 1 << 40
    ptrs = [base * (k + 1) for k in range(8)]
    # a gradient buffer overlapping an input is refused
    bad = list(ptrs)
    bad[6] = ptrs[1] + 64
    st, msg = _err(lambda: es.plan_backward(T, [4, 8, 32], 1, ptrs=bad))
    assert st == 3 and "overlaps" in msg
    # misaligned gradient buffer: generic path
    odd = list(ptrs)
    odd[7] = ptrs[7] + 4
    assert es.plan_backward(T, [4, 8, 32], 1, ptrs=odd)["path"] == "generic"
    # shapes are validated exactly as for the forward call
    assert _err(lambda: es.plan_backward(N, [2, 3, 4], 1))[0] == 4
    assert _err(lambda: es.plan_backward(T, [2, 3, 4], 5))[0] == 1
