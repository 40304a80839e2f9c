"""es_scan_host_f32 / es_scan_body_host_f32 through the C ABI without a GPU:
the checks that come before any CUDA call (null host pointers, the piece
count, the call's shapes), with stand-in device addresses."""
import ctypes

import numpy as np
import pytest

from element_scan_recurrences_gb300 import binding as es

P = ctypes.c_void_p
SHAPE = (4, 64, 8)
DEV = [(k + 1) << 44 for k in range(4)]      # initial_d, x_d, a_d, out_d: aligned, disjoint stand-ins


def _host():
    x = np.zeros(SHAPE, np.float32)
    a = np.zeros(SHAPE, np.float32)
    init = np.zeros((SHAPE[0], SHAPE[2]), np.float32)
    out = np.zeros(SHAPE, np.float32)
    return init, x, a, out


def _call(fn, body, init=True, seq0=True, out=True, chunks=0, axis=1, shape=SHAPE):
    h_init, h_x, h_a, h_out = _host()
    seqs_h = (P * 2)(h_x.ctypes.data if seq0 else None, h_a.ctypes.data)
    seqs_d = (P * 2)(DEV[1], DEV[2])
    shp = (ctypes.c_int64 * len(shape))(*shape)
    return fn(body, h_init.ctypes.data if init else None, seqs_h, 2, shp, len(shape), axis, 0, None, 0,
              h_out.ctypes.data if out else None, DEV[0], seqs_d, DEV[3], chunks, None)


@pytest.mark.parametrize("kind", ["builtin", "program"])
def test_host_entry_checks(kind):
    L = es.lib()
    if kind == "builtin":
        fn, body = L.es_scan_host_f32, es.TANH_DECAY
    else:
        prog = es.Body("(lambda (h x a) (tanh (+ x (* a h))))")
        fn, body = L.es_scan_body_host_f32, prog._h
    for kw in ({"init": False}, {"seq0": False}, {"out": False}, {"chunks": 65}, {"chunks": -1}):
        assert _call(fn, body, **kw) == 3, kw                 # ES_E_ARG
    # the call's own shape checks (an axis outside the rank)
    assert _call(fn, body, axis=3) in (1, 2), "axis"
    # and an empty call needs no GPU at all
    assert _call(fn, body, shape=(0, 64, 8)) == 0


def test_host_entry_null_program():
    L = es.lib()
    assert _call(L.es_scan_body_host_f32, None) == 3
