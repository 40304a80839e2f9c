"""Body programs through the C ABI without a GPU: the library rejects exactly
the bodies the oracle rejects, plans the documented paths, and every kernel a
body may use compiles for sm_103a (NVRTC runs on the host)."""
import numpy as np
import pytest

import body_cases
import body_pins
from element_scan_recurrences_gb300 import binding as es
from oracle.body import BodyError, scan_body


def _rejected_by_library(state_axis, W, widths, text):
    try:
        b = es.Body(text)
    except es.EsError as e:
        assert e.status == 7, e
        return True
    shape = [1, 2, W] if state_axis else [1, 2]
    try:
        b.plan(shape, 1, W if state_axis else 0, widths if state_axis else None)
    except es.EsError as e:
        return e.status in (1, 7)   # E-DIM-001 for a width that does not fit, else ES_E_BODY
    return False


@pytest.mark.parametrize("case", body_pins.REJECTED, ids=[r[3] for r in body_pins.REJECTED])
def test_library_rejects_what_the_oracle_rejects(case):
    state_axis, W, widths, text = case
    with pytest.raises(BodyError):
        scan_body(text, np.zeros((1, W) if state_axis else (1,), np.float32),
                  [np.zeros((1, 2, w) if state_axis else (1, 2), np.float32) for w in widths], axis=1,
                  state_axis=state_axis)
    assert _rejected_by_library(state_axis, W, widths, text), text


@pytest.mark.parametrize("cid", body_cases.CASE_IDS)
def test_library_accepts_the_test_bodies(cid):
    c = body_cases.case(cid)
    b = es.Body(c[1])
    W = c[2]
    n = b.n_seqs
    assert n == len(c[4])
    src = b.source(W, c[3])
    assert "struct EsBody" in src and ("kNS = %d;" % n) in src


def test_plan_paths():
    avg = es.Body("(lambda (h x) (+ (* 0.9 h) (* 0.1 x)))")
    assert avg.plan([4, 100, 256], 1)["path"] == "lane_tma"
    assert avg.plan([4, 100, 250], 1)["path"] == "generic"      # rows not a multiple of 16 bytes
    assert avg.plan([4, 100, 16], 1)["path"] == "generic"       # fewer than 32 lanes
    assert avg.plan([0, 10, 64], 1)["path"] == "empty"
    with pytest.raises(es.EsError) as e:
        avg.plan([4, 0, 64], 1)                                 # T = 0
    assert e.value.status == 1
    with pytest.raises(es.EsError) as e:                        # `out` overlaps the first sequence
        avg.plan([4, 10, 64], 1, ptrs=[1 << 44, 2 << 44, (2 << 44) + 64])
    assert e.value.status == 3
    p = es.Body("(lambda (h x y) (+ h x y))").plan([4, 10, 64], 1)
    assert p["seq_width"] == (1, 1) and p["O"] == 4 and p["T"] == 10 and p["J"] == 64
    # the sequence axis last: time innermost when rows are 16-byte multiples of >= 32 trips
    assert avg.plan([300, 100], -1)["path"] == "time_tma"
    assert avg.plan([300, 102], -1)["path"] == "generic"
    assert avg.plan([300, 16], -1)["path"] == "generic"
    # vector states of 2, 4, 8, 16 values with enough lanes per CTA
    nc = es.Body(body_cases.NORMCAP_TEXT)
    assert nc.plan([2, 70, 48, 16], 1, 16, [16, 1])["path"] == "vec_tma"
    assert nc.plan([2, 70, 48, 16], 1, 16, [16, 16])["path"] == "vec_tma"
    assert nc.plan([2, 70, 6, 16], 1, 16, [16, 1])["path"] == "generic"      # fewer lanes than a CTA holds
    assert nc.plan([2, 70, 50, 16], 1, 16, [16, 1])["path"] == "generic"     # gate rows not 16-byte multiples
    assert nc.plan([2, 70, 50, 16], 1, 16, [16, 16])["path"] == "vec_tma"
    assert nc.plan([2, 70, 48, 3], 1, 3, [3, 1])["path"] == "generic"        # odd widths
    es.set_path_override("vec_tma")
    try:
        with pytest.raises(es.EsError) as e:
            nc.plan([2, 70, 48, 3], 1, 3, [3, 1])
        assert e.value.status == 4
    finally:
        es.set_path_override("auto")


def test_arity_and_limits():
    b = es.Body("(lambda (h x) (+ h x))")
    lib = es.lib()
    import ctypes
    shp = (ctypes.c_int64 * 3)(2, 3, 4)
    seqs = (ctypes.c_void_p * 2)(1 << 44, 2 << 44)
    info = es.PlanInfo()
    st = lib.es_plan_body_f32(b._h, 3 << 44, seqs, 2, shp, 3, 1, 0, None, 0, 4 << 44, ctypes.byref(info))
    assert st == 7 and b"takes 1 sequence" in lib.es_last_error()
    nine = "(lambda (h a b c d e f g k m) (+ h a b c d e f g k m))"
    with pytest.raises(es.EsError) as e:
        es.Body(nine).plan([2, 3, 64], 1)
    assert e.value.status == 4          # more than ES_MAX_SEQS sequences


def test_kernels_compile_for_sm103a():
    """NVRTC compiles every kernel variant of each test body's signature."""
    for cid in ("tanh_decay", "eight_seqs", "count_logic", "normcap_w16", "normcap_w4_wide_gate", "centre_w4",
                "softsign_w2", "row_max_w8", "odd_width_w3", "width_one_state"):
        c = body_cases.case(cid)
        es.Body(c[1]).prepare(c[2], c[3])


def test_generated_functor_uses_ieee_operations():
    src = es.Body("(lambda (h x a) (tanh (+ x (* a h))))").source()
    assert "__fmul_rn(sw[1][e], h[e])" in src and "__fadd_rn(sw[0][e]" in src and "tanhf(" in src
    src = es.Body("(lambda (h x) (* 3.0 0.1 x))").source()
    # the numbers fold in double precision into one constant: f32(0.30000000000000004)
    bits = np.float32(3.0 * 0.1).view(np.uint32)
    assert ("0x%08xu" % bits) in src and src.count("__fmul_rn") == 1
