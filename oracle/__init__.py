"""CPU oracle for `element-scan` -- TEST INFRASTRUCTURE, not the product.

Only the test suite, ``__graft_entry__.smoke()`` and the bench's CPU-baseline
and reference arms may import this package.  The product path (the CUDA
library and its Python binding) never imports it and shares no code with it.

The arithmetic lives in ``es_oracle.c`` (a plain lane-by-lane loop, built with
``gcc -O2 -ffp-contract=off``); this module only compiles it and marshals numpy
arrays across ctypes.  ``scan_threads`` / ``scan_backward_threads`` run that
same loop on every host core, one contiguous block of lanes per thread.  Semantics follow "Nonlinear element scans"
(sx.041.io/docs/element-scan.md): intro (forward recurrence, output holds the
state after every trip), the `:state-axis` example (NORMCAP), the `:reverse`
paragraph (MAXPLUS, reverse order) and "Arguments and body" (shapes).
"""
from __future__ import annotations

import concurrent.futures
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "es_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libes_oracle.so")

TANH_DECAY = 0
NORMCAP = 1
MAXPLUS = 2
BODIES = {"TANH_DECAY": TANH_DECAY, "NORMCAP": NORMCAP, "MAXPLUS": MAXPLUS}

_lock = threading.Lock()
_lib = None

GCC_FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def compile_source(src: str, lib_path: str) -> str:
    """Compile an oracle source file into a shared library at ``lib_path``."""
    os.makedirs(os.path.dirname(lib_path), exist_ok=True)
    tmp = lib_path + ".%d.tmp" % os.getpid()
    subprocess.run(["gcc"] + GCC_FLAGS + ["-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, lib_path)
    return lib_path


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library (plain gcc, no fast-math)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


def _bind(lib_path: str):
    lib = ctypes.CDLL(lib_path)
    if hasattr(lib, "es_oracle_backward_f32"):
        fp = ctypes.POINTER(ctypes.c_float)
        fb = lib.es_oracle_backward_f32
        fb.restype = ctypes.c_int
        fb.argtypes = [ctypes.c_int, fp, ctypes.POINTER(fp), ctypes.c_int, ctypes.POINTER(ctypes.c_int64),
                       ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                       fp, fp, fp, ctypes.POINTER(fp)]
    for name, ft in (("es_oracle_f32", ctypes.c_float),
                     ("es_oracle_f64", ctypes.c_double)):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = [
            ctypes.c_int,                         # body
            ctypes.POINTER(ft),                   # initial
            ctypes.POINTER(ctypes.POINTER(ft)),   # seqs
            ctypes.c_int,                         # n_seqs
            ctypes.POINTER(ctypes.c_int64),       # shape
            ctypes.c_int,                         # rank
            ctypes.c_int,                         # axis
            ctypes.c_int,                         # state_width
            ctypes.POINTER(ctypes.c_int64),       # seq_widths or NULL
            ctypes.c_int,                         # reverse
            ctypes.POINTER(ft),                   # out
        ]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB_PATH)
    return _lib


def _body_id(body) -> int:
    if isinstance(body, str):
        return BODIES[body.upper()]
    return int(body)


def _c_array(a, dtype):
    """A C-contiguous array of `dtype` that keeps the rank (0-d stays 0-d)."""
    a = np.asarray(a, dtype=dtype)
    return a if a.flags.c_contiguous else a.copy(order="C")


def scan(body, initial, seqs, axis: int = 0, state_axis: bool = False,
         reverse: bool = False, dtype=np.float32, _lib=None, out=None) -> np.ndarray:
    """Run the oracle on host arrays and return the states after every trip.

    ``initial`` has the output shape with ``axis`` removed; ``seqs`` is a list
    of two arrays.  Without ``state_axis`` both have the output shape; with it,
    each may have its own last width (1 or the state width W).
    ``dtype=np.float64`` runs the double-precision diagnostic twin.  ``out``,
    when given, is a C-contiguous array of the output shape and dtype that
    receives the states (and is returned).
    """
    lib = _lib if _lib is not None else _load()
    ft = ctypes.c_float if dtype == np.float32 else ctypes.c_double
    fn = lib.es_oracle_f32 if dtype == np.float32 else lib.es_oracle_f64
    seqs = [_c_array(s, dtype) for s in seqs]
    initial = _c_array(initial, dtype)
    if len(seqs) != 2:
        raise ValueError("every body takes exactly two sequences")
    # output shape: the first sequence's shape; under a state axis its last
    # dim is the state width, which is initial's last dim
    shape = list(seqs[0].shape)
    rank = len(shape)
    if state_axis:
        if initial.ndim < 1 or rank < 2:
            raise ValueError("a state axis needs rank >= 2")
        shape[-1] = initial.shape[-1]
    W = shape[-1] if state_axis else 0
    ax = axis + rank if axis < 0 else axis
    if not 0 <= ax < rank:
        raise ValueError("axis %d out of range for rank %d" % (axis, rank))
    want_init = shape[:ax] + shape[ax + 1:]
    if list(initial.shape) != want_init:
        raise ValueError("initial shape %r, expected %r" % (list(initial.shape), want_init))
    for s in seqs:
        want = list(shape)
        if state_axis and s.ndim == rank and s.shape[-1] == 1:
            want[-1] = 1
        if list(s.shape) != want:
            raise ValueError("sequence shape %r, expected %r" % (list(s.shape), want))
    widths = None
    if state_axis:
        widths = (ctypes.c_int64 * 2)(*[s.shape[-1] for s in seqs])
    if out is None:
        out = np.empty(shape, dtype=dtype)
    elif list(out.shape) != shape or out.dtype != dtype or not out.flags.c_contiguous:
        raise ValueError("out must be a C-contiguous %s array of shape %r" % (np.dtype(dtype).name, shape))
    ptrs = (ctypes.POINTER(ft) * 2)(*[s.ctypes.data_as(ctypes.POINTER(ft)) for s in seqs])
    rc = fn(_body_id(body), initial.ctypes.data_as(ctypes.POINTER(ft)), ptrs, 2,
            (ctypes.c_int64 * rank)(*shape), rank, int(axis), int(W), widths,
            int(bool(reverse)), out.ctypes.data_as(ctypes.POINTER(ft)))
    if rc != 0:
        raise ValueError("oracle rejected arguments: body=%r shape=%r axis=%r state_axis=%r"
                         % (body, shape, axis, state_axis))
    return out


def scan_backward(body, initial, seqs, states, grad_out, axis: int = 0, state_axis: bool = False,
                  reverse: bool = False, _lib=None, out=None):
    """Gradients of sum(grad_out * scan(...)) with respect to initial and both
    sequences, from the forward states.  Returns (grad_initial, [gx, ga]) with
    the shapes of initial and of each sequence.  ``out``, when given, is
    (grad_initial, [gx, ga]): C-contiguous f32 arrays of those shapes that
    receive the gradients."""
    lib = _lib if _lib is not None else _load()
    ft = ctypes.c_float
    fp = ctypes.POINTER(ft)
    seqs = [_c_array(s, np.float32) for s in seqs]
    initial = _c_array(initial, np.float32)
    states = _c_array(states, np.float32)
    grad_out = _c_array(grad_out, np.float32)
    shape = list(states.shape)
    if list(grad_out.shape) != shape:
        raise ValueError("grad_out shape %r, expected %r" % (list(grad_out.shape), shape))
    rank = len(shape)
    W = shape[-1] if state_axis else 0
    ax = axis + rank if axis < 0 else axis
    if not 0 <= ax < rank:
        raise ValueError("axis out of range")
    if list(initial.shape) != shape[:ax] + shape[ax + 1:]:
        raise ValueError("initial shape %r does not fit %r" % (list(initial.shape), shape))
    for s in seqs:
        want = list(shape)
        if state_axis and s.shape[-1] == 1:
            want[-1] = 1
        if list(s.shape) != want:
            raise ValueError("sequence shape %r, expected %r" % (list(s.shape), want))
    widths = (ctypes.c_int64 * 2)(*[s.shape[-1] for s in seqs]) if state_axis else None
    if out is None:
        g_init = np.empty_like(initial)
        g_seqs = [np.empty_like(s) for s in seqs]
    else:
        g_init, g_seqs = out[0], list(out[1])
        for g, ref in zip([g_init] + g_seqs, [initial] + seqs):
            if g.shape != ref.shape or g.dtype != np.float32 or not g.flags.c_contiguous:
                raise ValueError("gradient buffers must be C-contiguous f32 arrays of the operands' shapes")
    sp = (fp * 2)(*[s.ctypes.data_as(fp) for s in seqs])
    gp = (fp * 2)(*[g.ctypes.data_as(fp) for g in g_seqs])
    rc = lib.es_oracle_backward_f32(_body_id(body), initial.ctypes.data_as(fp), sp, 2, (ctypes.c_int64 * rank)(*shape),
                                    rank, int(axis), int(W), widths, int(bool(reverse)), states.ctypes.data_as(fp),
                                    grad_out.ctypes.data_as(fp), g_init.ctypes.data_as(fp), gp)
    if rc != 0:
        raise ValueError("oracle rejected backward arguments")
    return g_init, g_seqs


class Oracle:
    """An oracle bound to one compiled library (tests load mutated builds)."""

    def __init__(self, lib_path: str):
        self._lib = _bind(lib_path)

    def scan(self, body, initial, seqs, axis: int = 0, state_axis: bool = False,
             reverse: bool = False, dtype=np.float32) -> np.ndarray:
        return scan(body, initial, seqs, axis=axis, state_axis=state_axis,
                    reverse=reverse, dtype=dtype, _lib=self._lib)

    def scan_backward(self, body, initial, seqs, states, grad_out, axis: int = 0, state_axis: bool = False,
                      reverse: bool = False):
        return scan_backward(body, initial, seqs, states, grad_out, axis=axis, state_axis=state_axis,
                             reverse=reverse, _lib=self._lib)


def scan_lanes(body, initial, x, a, reverse: bool = False) -> np.ndarray:
    """Scalar-state scan over independent lanes laid out as [L, T] rows.

    Convenience for sampled-lane parity: ``x`` and ``a`` are [L, T], ``initial``
    is [L]; the scan axis is 1.
    """
    return scan(body, initial, [x, a], axis=1, state_axis=False, reverse=reverse)


# ---------------------------------------------------------------------------
# all host cores: the same loop on contiguous blocks of lanes

def host_threads() -> int:
    """The host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _lane_blocks(dim0: int, threads: int):
    """Split [0, dim0) into at most `threads` contiguous blocks of nearly equal size."""
    k = max(1, min(threads, dim0))
    bounds = [dim0 * i // k for i in range(k + 1)]
    return [(bounds[i], bounds[i + 1]) for i in range(k) if bounds[i + 1] > bounds[i]]


def _run_blocks(jobs, threads: int):
    if len(jobs) == 1:
        jobs[0]()
        return
    # ctypes releases the interpreter lock for the duration of each call, so
    # the blocks run at the same time
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as pool:
        for f in [pool.submit(j) for j in jobs]:
            f.result()


def split_rows(fn, n_rows: int, threads: int = 0) -> int:
    """Call fn(lo, hi) on contiguous blocks of rows [0, n_rows), one thread a
    block (`host_threads()` blocks by default); for running any of the oracles
    on independent lanes at once.  Returns the number of blocks."""
    threads = threads or host_threads()
    blocks = _lane_blocks(n_rows, threads)
    _run_blocks([lambda lo=lo, hi=hi: fn(lo, hi) for lo, hi in blocks], threads)
    return len(blocks)


def scan_threads(body, initial, seqs, axis: int = 0, state_axis: bool = False, reverse: bool = False,
                 threads: int = 0) -> np.ndarray:
    """`scan` on every host core (f32): the lanes are split along dim 0 into
    contiguous blocks, and each block is scanned by the unchanged single-thread
    loop in a thread of its own, writing its slice of one output array.  Lanes
    are independent ("Nonlinear element scans", intro), so the result is the
    single-thread result bit for bit.  When the sequence axis is dim 0 (or
    there is one block) it is exactly `scan`.  ``threads`` = 0 takes
    `host_threads()`."""
    threads = threads or host_threads()
    seqs = [_c_array(s, np.float32) for s in seqs]
    initial = _c_array(initial, np.float32)
    rank = seqs[0].ndim
    ax = axis + rank if axis < 0 else axis
    if ax <= 0 or threads <= 1 or seqs[0].shape[0] <= 1:
        return scan(body, initial, seqs, axis=axis, state_axis=state_axis, reverse=reverse)
    shape = list(seqs[0].shape)
    if state_axis:
        shape[-1] = initial.shape[-1]
    # the whole call is checked once, on a view of no lanes along dim 0
    scan(body, initial[:0], [s[:0] for s in seqs], axis=axis, state_axis=state_axis, reverse=reverse)
    out = np.empty(shape, np.float32)
    lib = _load()
    jobs = [lambda lo=lo, hi=hi: scan(body, initial[lo:hi], [s[lo:hi] for s in seqs], axis=axis,
                                      state_axis=state_axis, reverse=reverse, _lib=lib, out=out[lo:hi])
            for lo, hi in _lane_blocks(shape[0], threads)]
    _run_blocks(jobs, threads)
    return out


def scan_backward_threads(body, initial, seqs, states, grad_out, axis: int = 0, state_axis: bool = False,
                          reverse: bool = False, threads: int = 0):
    """`scan_backward` on every host core, split into contiguous blocks of
    lanes along dim 0 exactly as `scan_threads`; each lane's gradient is its
    own reverse scan, so the result is the single-thread result bit for bit."""
    threads = threads or host_threads()
    seqs = [_c_array(s, np.float32) for s in seqs]
    initial = _c_array(initial, np.float32)
    states = _c_array(states, np.float32)
    grad_out = _c_array(grad_out, np.float32)
    rank = states.ndim
    ax = axis + rank if axis < 0 else axis
    if ax <= 0 or threads <= 1 or states.shape[0] <= 1:
        return scan_backward(body, initial, seqs, states, grad_out, axis=axis, state_axis=state_axis,
                             reverse=reverse)
    g_init = np.empty_like(initial)
    g_seqs = [np.empty_like(s) for s in seqs]
    lib = _load()
    jobs = [lambda lo=lo, hi=hi: scan_backward(body, initial[lo:hi], [s[lo:hi] for s in seqs], states[lo:hi],
                                               grad_out[lo:hi], axis=axis, state_axis=state_axis,
                                               reverse=reverse, _lib=lib,
                                               out=(g_init[lo:hi], [g[lo:hi] for g in g_seqs]))
            for lo, hi in _lane_blocks(states.shape[0], threads)]
    _run_blocks(jobs, threads)
    return g_init, g_seqs
