"""ctypes binding over libes.so (include/es.h).

Argument marshalling only: every step of a scan runs in the library's CUDA
kernels.  The binding raises ``LibraryMissing`` when libes.so has not been
built and ``EsError`` (with the library's message) for every non-OK status;
there is no CPU fallback.  Tensors are PyTorch CUDA tensors (PyTorch supplies
device memory and streams only).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

from . import build as _build

TANH_DECAY = 0
NORMCAP = 1
MAXPLUS = 2
_BODIES = {"TANH_DECAY": TANH_DECAY, "NORMCAP": NORMCAP, "MAXPLUS": MAXPLUS}

STATUS = {0: "ES_OK", 1: "ES_E_DIM_001", 2: "ES_E_DIM_002", 3: "ES_E_ARG", 4: "ES_E_UNSUPPORTED",
          5: "ES_E_CUDA", 6: "ES_E_TIMEOUT", 7: "ES_E_BODY"}
MAX_SEQS = 8
PATHS = {0: "auto", 1: "empty", 2: "generic", 3: "lane_tma", 4: "time_tma", 5: "vec_tma", 6: "mat_tma",
         7: "mat_chunked", 8: "mat_chunked_tma"}
PATH_IDS = {v: k for k, v in PATHS.items()}

# every function include/es.h declares
EXPORTS = ("es_scan_f32", "es_plan_f32", "es_scan_backward_f32", "es_plan_backward_f32", "es_device_status",
           "es_last_error", "es_status_string", "es_launch_count", "es_set_path_override", "es_set_wait_limit_ns",
           "es_set_drop_tile", "es_body_create", "es_body_destroy", "es_body_n_seqs", "es_scan_body_f32",
           "es_plan_body_f32", "es_body_source", "es_body_prepare", "es_body_compile_count", "es_matrix_scan_f32",
           "es_plan_matrix_scan_f32", "es_linear_scan_f32", "es_plan_linear_scan_f32", "es_table_scan_i32",
           "es_plan_table_scan_i32", "es_matrix_scan_workspace_f32", "es_matrix_scan_ws_f32",
           "es_plan_matrix_scan_ws_f32",
           "es_matrix_scan_static_f32", "es_scan_body_backward_f32", "es_plan_body_backward_f32",
           "es_body_source_backward", "es_body_prepare_backward", "es_matrix_scan_backward_f32",
           "es_plan_matrix_scan_backward_f32", "es_linear_scan_backward_f32", "es_plan_linear_scan_backward_f32",
           "es_scan_host_f32", "es_scan_body_host_f32", "es_matrix_scan_backward_ws_f32",
           "es_plan_matrix_scan_backward_ws_f32")


class LibraryMissing(ImportError):
    pass


class EsError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (STATUS.get(status, status), message))
        self.status = status
        self.message = message


class PlanInfo(ctypes.Structure):
    _fields_ = [("O", ctypes.c_int64), ("T", ctypes.c_int64), ("J", ctypes.c_int64), ("W", ctypes.c_int64),
                ("seq_width", ctypes.c_int64 * MAX_SEQS), ("elements", ctypes.c_int64), ("path", ctypes.c_int),
                ("reverse", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def lib():
    """Load libes.so (built in-tree); raise LibraryMissing if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            raise LibraryMissing("libes.so is not built (%s); run __graft_entry__.build() first" % path)
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64p = ctypes.POINTER(ctypes.c_int64)
        sig = [ctypes.c_int, P, ctypes.POINTER(P), ctypes.c_int, i64p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
               i64p, ctypes.c_int, P]
        L.es_scan_f32.argtypes = sig + [P]
        L.es_scan_f32.restype = ctypes.c_int
        L.es_plan_f32.argtypes = sig + [ctypes.POINTER(PlanInfo)]
        L.es_plan_f32.restype = ctypes.c_int
        bsig = sig[:-1] + [P, P, P, ctypes.POINTER(P)]     # ..., reverse, states, grad_out, grad_init, grad_seqs
        L.es_scan_backward_f32.argtypes = bsig + [P]
        L.es_scan_backward_f32.restype = ctypes.c_int
        L.es_plan_backward_f32.argtypes = bsig + [ctypes.POINTER(PlanInfo)]
        L.es_plan_backward_f32.restype = ctypes.c_int
        L.es_device_status.argtypes = [P]
        L.es_device_status.restype = ctypes.c_int
        L.es_last_error.argtypes = []
        L.es_last_error.restype = ctypes.c_char_p
        L.es_status_string.argtypes = [ctypes.c_int]
        L.es_status_string.restype = ctypes.c_char_p
        L.es_launch_count.argtypes = []
        L.es_launch_count.restype = ctypes.c_uint64
        L.es_set_path_override.argtypes = [ctypes.c_int]
        L.es_set_path_override.restype = ctypes.c_int
        L.es_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        L.es_set_wait_limit_ns.restype = ctypes.c_int
        L.es_set_drop_tile.argtypes = [ctypes.c_int64]
        L.es_set_drop_tile.restype = ctypes.c_int
        L.es_body_create.argtypes = [ctypes.c_char_p, ctypes.POINTER(P)]
        L.es_body_create.restype = ctypes.c_int
        L.es_body_destroy.argtypes = [P]
        L.es_body_destroy.restype = ctypes.c_int
        L.es_body_n_seqs.argtypes = [P]
        L.es_body_n_seqs.restype = ctypes.c_int
        bodysig = [P] + sig[1:]
        L.es_scan_body_f32.argtypes = bodysig + [P]
        L.es_scan_body_f32.restype = ctypes.c_int
        L.es_plan_body_f32.argtypes = bodysig + [ctypes.POINTER(PlanInfo)]
        L.es_plan_body_f32.restype = ctypes.c_int
        L.es_body_source.argtypes = [P, ctypes.c_int, ctypes.c_int, i64p, ctypes.c_char_p, ctypes.c_size_t,
                                     ctypes.POINTER(ctypes.c_size_t)]
        L.es_body_source.restype = ctypes.c_int
        L.es_body_prepare.argtypes = [P, ctypes.c_int, ctypes.c_int, i64p, ctypes.c_int]
        L.es_body_prepare.restype = ctypes.c_int
        hsig = sig[:-1] + [P, P, ctypes.POINTER(P), P, ctypes.c_int, P]   # ..., out_h, init_d, seqs_d, out_d, chunks, stream
        L.es_scan_host_f32.argtypes = hsig
        L.es_scan_host_f32.restype = ctypes.c_int
        L.es_scan_body_host_f32.argtypes = [P] + hsig[1:]
        L.es_scan_body_host_f32.restype = ctypes.c_int
        L.es_scan_body_backward_f32.argtypes = [P] + bsig[1:] + [P]
        L.es_scan_body_backward_f32.restype = ctypes.c_int
        L.es_plan_body_backward_f32.argtypes = [P] + bsig[1:] + [ctypes.POINTER(PlanInfo)]
        L.es_plan_body_backward_f32.restype = ctypes.c_int
        L.es_body_source_backward.argtypes = [P, ctypes.c_int, ctypes.c_int, i64p, ctypes.c_char_p, ctypes.c_size_t,
                                              ctypes.POINTER(ctypes.c_size_t)]
        L.es_body_source_backward.restype = ctypes.c_int
        L.es_body_prepare_backward.argtypes = [P, ctypes.c_int, ctypes.c_int, i64p]
        L.es_body_prepare_backward.restype = ctypes.c_int
        L.es_body_compile_count.argtypes = []
        L.es_body_compile_count.restype = ctypes.c_uint64
        msig = [P, i64p, ctypes.c_int, P, i64p, ctypes.c_int, ctypes.c_int, ctypes.c_int]   # a, b, axis, reverse
        L.es_matrix_scan_f32.argtypes = msig + [ctypes.c_int, P, P]
        L.es_matrix_scan_f32.restype = ctypes.c_int
        L.es_plan_matrix_scan_f32.argtypes = msig + [ctypes.c_int, P, ctypes.POINTER(PlanInfo)]
        L.es_plan_matrix_scan_f32.restype = ctypes.c_int
        L.es_linear_scan_f32.argtypes = msig + [P, P]
        L.es_linear_scan_f32.restype = ctypes.c_int
        L.es_plan_linear_scan_f32.argtypes = msig + [P, ctypes.POINTER(PlanInfo)]
        L.es_plan_linear_scan_f32.restype = ctypes.c_int
        L.es_matrix_scan_workspace_f32.argtypes = [i64p, ctypes.c_int, i64p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   ctypes.POINTER(ctypes.c_size_t)]
        L.es_matrix_scan_workspace_f32.restype = ctypes.c_int
        L.es_matrix_scan_ws_f32.argtypes = msig + [ctypes.c_int, P, P, ctypes.c_size_t, P]
        L.es_matrix_scan_ws_f32.restype = ctypes.c_int
        L.es_plan_matrix_scan_ws_f32.argtypes = msig + [ctypes.c_int, P, P, ctypes.c_size_t,
                                                        ctypes.POINTER(PlanInfo)]
        L.es_plan_matrix_scan_ws_f32.restype = ctypes.c_int
        L.es_matrix_scan_static_f32.argtypes = msig + [ctypes.c_int, P, P]
        # ..., projective, states, grad_out, grad_a, grad_b
        L.es_matrix_scan_backward_f32.argtypes = msig + [ctypes.c_int, P, P, P, P, P]
        L.es_matrix_scan_backward_f32.restype = ctypes.c_int
        L.es_plan_matrix_scan_backward_f32.argtypes = msig + [ctypes.c_int, P, P, P, P, ctypes.POINTER(PlanInfo)]
        L.es_plan_matrix_scan_backward_f32.restype = ctypes.c_int
        L.es_matrix_scan_backward_ws_f32.argtypes = msig + [ctypes.c_int, P, P, P, P, P, ctypes.c_size_t, P]
        L.es_matrix_scan_backward_ws_f32.restype = ctypes.c_int
        L.es_plan_matrix_scan_backward_ws_f32.argtypes = msig + [ctypes.c_int, P, P, P, P, P, ctypes.c_size_t,
                                                                 ctypes.POINTER(PlanInfo)]
        L.es_plan_matrix_scan_backward_ws_f32.restype = ctypes.c_int
        L.es_linear_scan_backward_f32.argtypes = msig + [P, P, P, P, P]
        L.es_linear_scan_backward_f32.restype = ctypes.c_int
        L.es_plan_linear_scan_backward_f32.argtypes = msig + [P, P, P, P, ctypes.POINTER(PlanInfo)]
        L.es_plan_linear_scan_backward_f32.restype = ctypes.c_int
        L.es_matrix_scan_static_f32.restype = ctypes.c_int
        tsig = [P, ctypes.c_int64, ctypes.c_int64, P, i64p, ctypes.c_int, ctypes.c_int, ctypes.c_int32]
        L.es_table_scan_i32.argtypes = tsig + [P, P]
        L.es_table_scan_i32.restype = ctypes.c_int
        L.es_plan_table_scan_i32.argtypes = tsig + [P, ctypes.POINTER(PlanInfo)]
        L.es_plan_table_scan_i32.restype = ctypes.c_int
        _lib = L
        return L


def _check(status: int):
    if status != 0:
        raise EsError(status, lib().es_last_error().decode(errors="replace"))


def status_string(status: int) -> str:
    return lib().es_status_string(int(status)).decode()


def _body_id(body) -> int:
    if isinstance(body, str):
        return _BODIES[body.upper()]
    return int(body)


def _args(body, shape, axis, state_width, seq_widths):
    rank = len(shape)
    shp = (ctypes.c_int64 * max(rank, 1))(*shape)
    sw = None if seq_widths is None else (ctypes.c_int64 * 2)(*seq_widths)
    return _body_id(body), shp, rank, int(axis), int(state_width), sw


def plan(body, shape: Sequence[int], axis: int, state_width: int = 0, seq_widths=None, reverse: bool = False,
         ptrs: Optional[Sequence[int]] = None) -> dict:
    """Validate and plan a call without touching a GPU (pure host logic).

    ``ptrs`` are the (initial, x, second, out) addresses to plan for; by
    default 16-byte aligned, non-overlapping stand-ins.  Raises EsError for an
    invalid call, else returns the canonical view and the kernel path.
    """
    b, shp, rank, ax, sw_, widths = _args(body, shape, axis, state_width, seq_widths)
    if ptrs is None:
        ptrs = [(k + 1) << 44 for k in range(4)]
    seqs = (ctypes.c_void_p * 2)(ptrs[1], ptrs[2])
    info = PlanInfo()
    _check(lib().es_plan_f32(b, ptrs[0], seqs, 2, shp, rank, ax, sw_, widths, int(bool(reverse)), ptrs[3],
                             ctypes.byref(info)))
    return {"O": info.O, "T": info.T, "J": info.J, "W": info.W, "seq_width": (info.seq_width[0], info.seq_width[1]),
            "elements": info.elements, "path": PATHS[info.path], "reverse": bool(info.reverse)}


def _out_shape(initial, seqs, axis, state_axis):
    shape = list(seqs[0].shape)
    if state_axis:
        shape[-1] = initial.shape[-1]
    return shape


def _require_cuda_f32(t, name):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
        raise TypeError("%s must be a contiguous float32 CUDA tensor (got %s %s, contiguous=%s)"
                        % (name, t.device, t.dtype, t.is_contiguous()))


def scan(body, initial, seqs, axis: int = 0, state_axis: bool = False, reverse: bool = False, out=None,
         stream=None):
    """Run one element scan on CUDA tensors; returns ``out`` (allocated if None).

    ``seqs`` is ``[x, a]`` (TANH_DECAY, NORMCAP) or ``[x, c]`` (MAXPLUS).  The
    call is asynchronous on ``stream`` (default: PyTorch's current stream).
    """
    import torch
    seqs = list(seqs)
    if len(seqs) != 2:
        raise EsError(3, "every body takes exactly two sequences")
    _require_cuda_f32(initial, "initial")
    for k, s in enumerate(seqs):
        _require_cuda_f32(s, "sequence %d" % k)
    shape = _out_shape(initial, seqs, axis, state_axis)
    if out is None:
        out = torch.empty(shape, device=seqs[0].device, dtype=torch.float32)
    else:
        _require_cuda_f32(out, "out")
        if list(out.shape) != shape:
            raise EsError(1, "out shape %s does not match the output shape %s" % (list(out.shape), shape))
    return scan_into(body, initial, seqs, out, axis=axis, state_axis=state_axis, reverse=reverse, stream=stream)


def scan_into(body, initial, seqs, out, axis: int = 0, state_axis: bool = False, reverse: bool = False,
              stream=None):
    """es_scan_f32 on tensors the caller has already checked (no allocation)."""
    import torch
    shape = list(out.shape)
    state_width = shape[-1] if state_axis else 0
    seq_widths = [int(s.shape[-1]) for s in seqs] if state_axis else None
    b, shp, rank, ax, sw_, widths = _args(body, shape, axis, state_width, seq_widths)
    ptrs = (ctypes.c_void_p * 2)(seqs[0].data_ptr(), seqs[1].data_ptr())
    if stream is None:
        stream = torch.cuda.current_stream(out.device)
    handle = stream if isinstance(stream, int) else stream.cuda_stream
    _check(lib().es_scan_f32(b, initial.data_ptr(), ptrs, 2, shp, rank, ax, sw_, widths, int(bool(reverse)),
                             out.data_ptr(), handle))
    return out


def _host_args(initial_h, seqs_h, out_h, dev_bufs):
    init_d, seqs_d, out_d = dev_bufs
    for t, nm in [(initial_h, "initial_h"), (out_h, "out_h")] + [(h, "sequence %d" % k) for k, h in enumerate(seqs_h)]:
        if t.is_cuda or not t.is_contiguous() or str(t.dtype) != "torch.float32":
            raise TypeError("%s must be a contiguous float32 host tensor" % nm)
    _require_cuda_f32(init_d, "initial_d")
    _require_cuda_f32(out_d, "out_d")
    for k, d in enumerate(seqs_d):
        _require_cuda_f32(d, "device sequence %d" % k)
    n = len(seqs_h)
    hp = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in seqs_h])
    dp = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in seqs_d])
    return init_d, out_d, hp, dp


def scan_host(body, initial_h, seqs_h, out_h, dev_bufs, axis: int = 0, state_axis: bool = False,
              reverse: bool = False, stream=None, chunks: int = 0):
    """End-to-end call on host tensors (es_scan_host_f32): the library copies
    the inputs from (pinned) host memory into the caller's device buffers,
    scans and copies the states back, in row pieces that overlap.

    ``dev_bufs`` = (initial_d, [x_d, a_d], out_d), preallocated by the caller.
    Asynchronous on ``stream``; synchronise before reading ``out_h``.
    """
    import torch
    init_d, out_d, hp, dp = _host_args(initial_h, seqs_h, out_h, dev_bufs)
    shape = list(out_h.shape)
    state_width = shape[-1] if state_axis else 0
    seq_widths = [int(t.shape[-1]) for t in seqs_h] if state_axis else None
    b, shp, rank, ax, sw_, widths = _args(body, shape, axis, state_width, seq_widths)
    if stream is None:
        stream = torch.cuda.current_stream(out_d.device)
    handle = stream if isinstance(stream, int) else stream.cuda_stream
    _check(lib().es_scan_host_f32(b, initial_h.data_ptr(), hp, len(seqs_h), shp, rank, ax, sw_, widths,
                                  int(bool(reverse)), out_h.data_ptr(), init_d.data_ptr(), dp, out_d.data_ptr(),
                                  int(chunks), handle))
    return out_h


def plan_backward(body, shape: Sequence[int], axis: int, state_width: int = 0, seq_widths=None,
                  reverse: bool = False, ptrs: Optional[Sequence[int]] = None) -> dict:
    """Validate and plan a backward call without a GPU.  ``ptrs`` are the
    (initial, x, second, states, grad_out, grad_initial, grad_x, grad_second)
    addresses; by default 16-byte aligned, non-overlapping stand-ins."""
    b, shp, rank, ax, sw_, widths = _args(body, shape, axis, state_width, seq_widths)
    if ptrs is None:
        ptrs = [(k + 1) << 44 for k in range(8)]
    seqs = (ctypes.c_void_p * 2)(ptrs[1], ptrs[2])
    gseqs = (ctypes.c_void_p * 2)(ptrs[6], ptrs[7])
    info = PlanInfo()
    _check(lib().es_plan_backward_f32(b, ptrs[0], seqs, 2, shp, rank, ax, sw_, widths, int(bool(reverse)), ptrs[3],
                                      ptrs[4], ptrs[5], gseqs, ctypes.byref(info)))
    return {"O": info.O, "T": info.T, "J": info.J, "W": info.W, "seq_width": (info.seq_width[0], info.seq_width[1]),
            "elements": info.elements, "path": PATHS[info.path], "reverse": bool(info.reverse)}


def scan_backward(body, initial, seqs, states, grad_out, axis: int = 0, state_axis: bool = False,
                  reverse: bool = False, grads=None, stream=None):
    """Gradients of sum(grad_out * scan(...)) on CUDA tensors.

    ``states`` is the forward output.  Returns (grad_initial, [grad_x,
    grad_second]) shaped like initial and the two sequences; ``grads`` may
    supply those buffers.  Asynchronous on ``stream``.
    """
    import torch
    seqs = list(seqs)
    _require_cuda_f32(initial, "initial")
    for k, t in enumerate(seqs):
        _require_cuda_f32(t, "sequence %d" % k)
    _require_cuda_f32(states, "states")
    _require_cuda_f32(grad_out, "grad_out")
    shape = list(states.shape)
    if list(grad_out.shape) != shape:
        raise EsError(1, "grad_out shape %s does not match the states %s" % (list(grad_out.shape), shape))
    if grads is None:
        grads = (torch.empty_like(initial), [torch.empty_like(t) for t in seqs])
    g_init, g_seqs = grads
    for t in [g_init] + list(g_seqs):
        _require_cuda_f32(t, "gradient buffer")
    state_width = shape[-1] if state_axis else 0
    seq_widths = [int(t.shape[-1]) for t in seqs] if state_axis else None
    b, shp, rank, ax, sw_, widths = _args(body, shape, axis, state_width, seq_widths)
    sp = (ctypes.c_void_p * 2)(seqs[0].data_ptr(), seqs[1].data_ptr())
    gp = (ctypes.c_void_p * 2)(g_seqs[0].data_ptr(), g_seqs[1].data_ptr())
    if stream is None:
        stream = torch.cuda.current_stream(states.device)
    handle = stream if isinstance(stream, int) else stream.cuda_stream
    _check(lib().es_scan_backward_f32(b, initial.data_ptr(), sp, 2, shp, rank, ax, sw_, widths, int(bool(reverse)),
                                      states.data_ptr(), grad_out.data_ptr(), g_init.data_ptr(), gp, handle))
    return g_init, list(g_seqs)


def device_status(stream=None):
    """Synchronise and raise EsError(ES_E_TIMEOUT) if a kernel gave up a wait."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream if isinstance(stream, int) else stream.cuda_stream
    _check(lib().es_device_status(handle))


def launch_count() -> int:
    return int(lib().es_launch_count())


def set_path_override(path) -> None:
    _check(lib().es_set_path_override(PATH_IDS[path] if isinstance(path, str) else int(path)))


def set_wait_limit_ns(ns: int) -> None:
    _check(lib().es_set_wait_limit_ns(int(ns)))


def set_drop_tile(k: int) -> None:
    _check(lib().es_set_drop_tile(int(k)))


# ---------------------------------------------------------------------------
# body programs


def _widths_array(seq_widths):
    if seq_widths is None:
        return None
    return (ctypes.c_int64 * max(len(seq_widths), 1))(*[int(w) for w in seq_widths])


class Body:
    """A body program: an element-scan body given as text in the pages'
    lambda notation, e.g. ``(lambda (h x a) (tanh (+ x (* a h))))``.

    Created (read and checked) by libes.so; each call signature is compiled
    into a CUDA kernel at run time on first use.  Raises EsError
    (ES_E_BODY) for a body the contract rejects.
    """

    def __init__(self, text: str):
        handle = ctypes.c_void_p()
        _check(lib().es_body_create(text.encode(), ctypes.byref(handle)))
        self._h = handle
        self.text = text

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value is not None and _lib is not None:
            _lib.es_body_destroy(h)
            self._h = None

    @property
    def n_seqs(self) -> int:
        return int(lib().es_body_n_seqs(self._h))

    def source(self, state_width: int = 0, seq_widths=None) -> str:
        """The CUDA functor generated for a signature."""
        n = self.n_seqs
        sw = _widths_array(seq_widths)
        need = ctypes.c_size_t()
        _check(lib().es_body_source(self._h, int(state_width), n, sw, None, 0, ctypes.byref(need)))
        buf = ctypes.create_string_buffer(need.value + 1)
        _check(lib().es_body_source(self._h, int(state_width), n, sw, buf, need.value + 1, ctypes.byref(need)))
        return buf.value.decode()

    def source_backward(self, state_width: int = 0, seq_widths=None) -> str:
        """The functor with its vector-Jacobian product for a signature."""
        n = self.n_seqs
        sw = _widths_array(seq_widths)
        need = ctypes.c_size_t()
        _check(lib().es_body_source_backward(self._h, int(state_width), n, sw, None, 0, ctypes.byref(need)))
        buf = ctypes.create_string_buffer(need.value + 1)
        _check(lib().es_body_source_backward(self._h, int(state_width), n, sw, buf, need.value + 1,
                                             ctypes.byref(need)))
        return buf.value.decode()

    def vjp_live_mask(self, state_width: int = 0, seq_widths=None) -> int:
        """Bit k set when the body's vector-Jacobian product reads sequence k
        (the others are not streamed by the backward kernels)."""
        src = self.source_backward(state_width, seq_widths)
        key = "kVjpSeqs = 0x"
        at = src.index(key) + len(key)
        return int(src[at:src.index("u", at)], 16)

    def prepare_backward(self, state_width: int = 0, seq_widths=None) -> None:
        """Compile ahead of time the backward kernel of a signature (no GPU needed)."""
        _check(lib().es_body_prepare_backward(self._h, int(state_width), self.n_seqs, _widths_array(seq_widths)))

    def plan_backward(self, shape: Sequence[int], axis: int, state_width: int = 0, seq_widths=None,
                      reverse: bool = False, ptrs: Optional[Sequence[int]] = None) -> dict:
        """Validate and plan a backward call without a GPU.  ``ptrs`` are
        (initial, seq 0 .. seq n-1, states, grad_out, grad_initial, grad seq
        0 .. n-1); by default 16-byte aligned, non-overlapping stand-ins."""
        n = self.n_seqs
        rank = len(shape)
        shp = (ctypes.c_int64 * max(rank, 1))(*shape)
        if ptrs is None:
            ptrs = [(k + 1) << 44 for k in range(2 * n + 4)]
        seqs = (ctypes.c_void_p * n)(*ptrs[1:n + 1])
        gseqs = (ctypes.c_void_p * n)(*ptrs[n + 4:2 * n + 4])
        info = PlanInfo()
        _check(lib().es_plan_body_backward_f32(self._h, ptrs[0], seqs, n, shp, rank, int(axis), int(state_width),
                                               _widths_array(seq_widths), int(bool(reverse)), ptrs[n + 1],
                                               ptrs[n + 2], ptrs[n + 3], gseqs, ctypes.byref(info)))
        return {"O": info.O, "T": info.T, "J": info.J, "W": info.W,
                "seq_width": tuple(info.seq_width[k] for k in range(n)), "elements": info.elements,
                "path": PATHS[info.path], "reverse": bool(info.reverse)}

    def scan_backward(self, initial, seqs, states, grad_out, axis: int = 0, state_axis: bool = False,
                      reverse: bool = False, grads=None, stream=None):
        """Gradients of sum(grad_out * scan(...)) on CUDA tensors.

        ``states`` is the forward output.  Returns (grad_initial, [grad seq
        k]) shaped like initial and the sequences; ``grads`` may supply those
        buffers.  Asynchronous on ``stream``."""
        import torch
        seqs = list(seqs)
        _require_cuda_f32(initial, "initial")
        for k, t in enumerate(seqs):
            _require_cuda_f32(t, "sequence %d" % k)
        _require_cuda_f32(states, "states")
        _require_cuda_f32(grad_out, "grad_out")
        shape = list(states.shape)
        if list(grad_out.shape) != shape:
            raise EsError(1, "grad_out shape %s does not match the states %s" % (list(grad_out.shape), shape))
        if grads is None:
            grads = (torch.empty_like(initial), [torch.empty_like(t) for t in seqs])
        g_init, g_seqs = grads
        for t in [g_init] + list(g_seqs):
            _require_cuda_f32(t, "gradient buffer")
        n = len(seqs)
        rank = len(shape)
        shp = (ctypes.c_int64 * max(rank, 1))(*shape)
        state_width = shape[-1] if state_axis else 0
        sw = _widths_array([int(t.shape[-1]) for t in seqs]) if state_axis else None
        sp = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in seqs])
        gp = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in g_seqs])
        if stream is None:
            stream = torch.cuda.current_stream(states.device)
        handle = stream if isinstance(stream, int) else stream.cuda_stream
        _check(lib().es_scan_body_backward_f32(self._h, initial.data_ptr(), sp, n, shp, rank, int(axis),
                                               int(state_width), sw, int(bool(reverse)), states.data_ptr(),
                                               grad_out.data_ptr(), g_init.data_ptr(), gp, handle))
        return g_init, list(g_seqs)

    def prepare(self, state_width: int = 0, seq_widths=None, path="auto") -> None:
        """Compile ahead of time the kernels a signature may use (no GPU needed)."""
        p = PATH_IDS[path] if isinstance(path, str) else int(path)
        _check(lib().es_body_prepare(self._h, int(state_width), self.n_seqs, _widths_array(seq_widths), p))

    def plan(self, shape: Sequence[int], axis: int, state_width: int = 0, seq_widths=None, reverse: bool = False,
             ptrs: Optional[Sequence[int]] = None) -> dict:
        """Validate and plan a call without a GPU (no kernel is compiled).
        ``ptrs`` are (initial, seq 0, ..., out); by default 16-byte aligned,
        non-overlapping stand-ins."""
        n = self.n_seqs
        rank = len(shape)
        shp = (ctypes.c_int64 * max(rank, 1))(*shape)
        if ptrs is None:
            ptrs = [(k + 1) << 44 for k in range(n + 2)]
        seqs = (ctypes.c_void_p * n)(*ptrs[1:n + 1])
        info = PlanInfo()
        _check(lib().es_plan_body_f32(self._h, ptrs[0], seqs, n, shp, rank, int(axis), int(state_width),
                                      _widths_array(seq_widths), int(bool(reverse)), ptrs[n + 1],
                                      ctypes.byref(info)))
        return {"O": info.O, "T": info.T, "J": info.J, "W": info.W,
                "seq_width": tuple(info.seq_width[k] for k in range(n)), "elements": info.elements,
                "path": PATHS[info.path], "reverse": bool(info.reverse)}

    def scan(self, initial, seqs, axis: int = 0, state_axis: bool = False, reverse: bool = False, out=None,
             stream=None):
        """Run the scan on CUDA tensors; returns ``out`` (allocated if None)."""
        import torch
        seqs = list(seqs)
        _require_cuda_f32(initial, "initial")
        for k, t in enumerate(seqs):
            _require_cuda_f32(t, "sequence %d" % k)
        if state_axis:
            wide = [t for t in seqs if t.shape[-1] == initial.shape[-1]]
            shape = list((wide[0] if wide else seqs[0]).shape[:-1]) + [int(initial.shape[-1])]
        else:
            shape = list(seqs[0].shape)
        if out is None:
            out = torch.empty(shape, device=seqs[0].device, dtype=torch.float32)
        else:
            _require_cuda_f32(out, "out")
            if list(out.shape) != shape:
                raise EsError(1, "out shape %s does not match the output shape %s" % (list(out.shape), shape))
        return self.scan_into(initial, seqs, out, axis=axis, state_axis=state_axis, reverse=reverse, stream=stream)

    def scan_into(self, initial, seqs, out, axis: int = 0, state_axis: bool = False, reverse: bool = False,
                  stream=None):
        """es_scan_body_f32 on tensors the caller has already checked."""
        import torch
        shape = list(out.shape)
        n = len(seqs)
        rank = len(shape)
        shp = (ctypes.c_int64 * max(rank, 1))(*shape)
        state_width = shape[-1] if state_axis else 0
        sw = _widths_array([int(t.shape[-1]) for t in seqs]) if state_axis else None
        ptrs = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in seqs])
        if stream is None:
            stream = torch.cuda.current_stream(out.device)
        handle = stream if isinstance(stream, int) else stream.cuda_stream
        _check(lib().es_scan_body_f32(self._h, initial.data_ptr(), ptrs, n, shp, rank, int(axis), int(state_width),
                                      sw, int(bool(reverse)), out.data_ptr(), handle))
        return out

    def scan_host(self, initial_h, seqs_h, out_h, dev_bufs, axis: int = 0, state_axis: bool = False,
                  reverse: bool = False, stream=None, chunks: int = 0):
        """End-to-end call on host tensors (es_scan_body_host_f32; see the
        module's ``scan_host``).  Asynchronous on ``stream``; synchronise
        before reading ``out_h``."""
        import torch
        init_d, out_d, hp, dp = _host_args(initial_h, seqs_h, out_h, dev_bufs)
        shape = list(out_h.shape)
        n = len(seqs_h)
        rank = len(shape)
        shp = (ctypes.c_int64 * max(rank, 1))(*shape)
        state_width = shape[-1] if state_axis else 0
        sw = _widths_array([int(t.shape[-1]) for t in seqs_h]) if state_axis else None
        if stream is None:
            stream = torch.cuda.current_stream(out_d.device)
        handle = stream if isinstance(stream, int) else stream.cuda_stream
        _check(lib().es_scan_body_host_f32(self._h, initial_h.data_ptr(), hp, n, shp, rank, int(axis),
                                           int(state_width), sw, int(bool(reverse)), out_h.data_ptr(),
                                           init_d.data_ptr(), dp, out_d.data_ptr(), int(chunks), handle))
        return out_h


def body_compile_count() -> int:
    return int(lib().es_body_compile_count())


# ---------------------------------------------------------------------------
# matrix-scan and linear-scan


def _shape_array(shape):
    shape = [int(d) for d in shape]
    return (ctypes.c_int64 * max(len(shape), 1))(*shape), len(shape)


def _lead_broadcast(sa, sb):
    r = max(len(sa), len(sb))
    sa = [1] * (r - len(sa)) + list(sa)
    sb = [1] * (r - len(sb)) + list(sb)
    return [y if x == 1 else x for x, y in zip(sa, sb)]


def _info(info, path_names=PATHS):
    return {"O": info.O, "T": info.T, "J": info.J, "W": info.W,
            "seq_width": (info.seq_width[0], info.seq_width[1]), "elements": info.elements,
            "path": path_names[info.path], "reverse": bool(info.reverse)}


def plan_matrix_scan(a_shape, b_shape, axis: int = 0, reverse: bool = False, projective: bool = False,
                     ptrs: Optional[Sequence[int]] = None) -> dict:
    """Validate and plan a matrix-scan without a GPU.  ``ptrs`` = (a, b, out),
    by default 16-byte aligned, non-overlapping stand-ins."""
    if ptrs is None:
        ptrs = [(k + 1) << 44 for k in range(3)]
    sa, ra = _shape_array(a_shape)
    sb, rb = _shape_array(b_shape)
    info = PlanInfo()
    _check(lib().es_plan_matrix_scan_f32(ptrs[0], sa, ra, ptrs[1], sb, rb, int(axis), int(bool(reverse)),
                                         int(bool(projective)), ptrs[2], ctypes.byref(info)))
    return _info(info)


def matrix_scan(a, b, axis: int = 0, reverse: bool = False, projective: bool = False, out=None, stream=None):
    """matrix-scan on CUDA tensors: h[t] = a[t] @ h[t-1] + b[t] along `axis`
    of the (broadcast) leading dims, from h = 0; returns ``out``."""
    import torch
    _require_cuda_f32(a, "a")
    _require_cuda_f32(b, "b")
    if a.dim() < 2 or b.dim() < 2:
        raise EsError(1, "a is [.., n, n] and b [.., n, m]")
    shape = _lead_broadcast(list(a.shape[:-2]), list(b.shape[:-2])) + [int(b.shape[-2]), int(b.shape[-1])]
    if out is None:
        out = torch.empty(shape, device=b.device, dtype=torch.float32)
    else:
        _require_cuda_f32(out, "out")
    sa, ra = _shape_array(a.shape)
    sb, rb = _shape_array(b.shape)
    if stream is None:
        stream = torch.cuda.current_stream(b.device)
    handle = stream if isinstance(stream, int) else stream.cuda_stream
    _check(lib().es_matrix_scan_f32(a.data_ptr(), sa, ra, b.data_ptr(), sb, rb, int(axis), int(bool(reverse)),
                                    int(bool(projective)), out.data_ptr(), handle))
    return out


def matrix_scan_workspace(a_shape, b_shape, axis: int = 0, projective: bool = False) -> int:
    """Workspace bytes the chunked path would use for these shapes (0: the
    call runs lane by lane and needs none).  No GPU needed."""
    sa, ra = _shape_array(a_shape)
    sb, rb = _shape_array(b_shape)
    n = ctypes.c_size_t()
    _check(lib().es_matrix_scan_workspace_f32(sa, ra, sb, rb, int(axis), int(bool(projective)), ctypes.byref(n)))
    return int(n.value)


def plan_matrix_scan_ws(a_shape, b_shape, workspace_bytes: int, axis: int = 0, reverse: bool = False,
                        projective: bool = False, ptrs: Optional[Sequence[int]] = None) -> dict:
    """The checks and the kernel path of ``matrix_scan_ws`` with a workspace
    of ``workspace_bytes``, without a GPU.  ``ptrs`` = (a, b, out, workspace),
    by default 16-byte aligned, non-overlapping stand-ins."""
    if ptrs is None:
        ptrs = [(k + 1) << 44 for k in range(4)]
    sa, ra = _shape_array(a_shape)
    sb, rb = _shape_array(b_shape)
    info = PlanInfo()
    _check(lib().es_plan_matrix_scan_ws_f32(ptrs[0], sa, ra, ptrs[1], sb, rb, int(axis), int(bool(reverse)),
                                            int(bool(projective)), ptrs[2], ptrs[3] if workspace_bytes else None,
                                            int(workspace_bytes), ctypes.byref(info)))
    return _info(info)


def matrix_scan_ws(a, b, workspace, axis: int = 0, reverse: bool = False, projective: bool = False, out=None,
                   stream=None):
    """matrix-scan with a caller workspace (a CUDA tensor of at least
    ``matrix_scan_workspace`` bytes): few long lanes run the chunked scan."""
    import torch
    _require_cuda_f32(a, "a")
    _require_cuda_f32(b, "b")
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda:
        raise TypeError("workspace must be a CUDA tensor")
    shape = _lead_broadcast(list(a.shape[:-2]), list(b.shape[:-2])) + [int(b.shape[-2]), int(b.shape[-1])]
    if out is None:
        out = torch.empty(shape, device=b.device, dtype=torch.float32)
    sa, ra = _shape_array(a.shape)
    sb, rb = _shape_array(b.shape)
    if stream is None:
        stream = torch.cuda.current_stream(b.device)
    handle = stream if isinstance(stream, int) else stream.cuda_stream
    _check(lib().es_matrix_scan_ws_f32(a.data_ptr(), sa, ra, b.data_ptr(), sb, rb, int(axis), int(bool(reverse)),
                                       int(bool(projective)), out.data_ptr(), workspace.data_ptr(),
                                       workspace.numel() * workspace.element_size(), handle))
    return out


STATIC_SCRATCH_BYTES = 32 << 20


def matrix_scan_static(a, b, axis: int = 0, reverse: bool = False, projective: bool = False, out=None,
                       stream=None):
    """es_matrix_scan_static_f32: matrix-scan whose chunked path (few long
    lanes) runs in the library's own static device scratch of
    STATIC_SCRATCH_BYTES, for callers that cannot allocate device memory.  A
    scan that would need more scratch raises EsError (ES_E_UNSUPPORTED).
    When ``out`` is None this wrapper allocates it with torch; a caller that
    may not allocate passes ``out``."""
    import torch
    _require_cuda_f32(a, "a")
    _require_cuda_f32(b, "b")
    shape = _lead_broadcast(list(a.shape[:-2]), list(b.shape[:-2])) + [int(b.shape[-2]), int(b.shape[-1])]
    if out is None:
        out = torch.empty(shape, device=b.device, dtype=torch.float32)
    sa, ra = _shape_array(a.shape)
    sb, rb = _shape_array(b.shape)
    if stream is None:
        stream = torch.cuda.current_stream(b.device)
    handle = stream if isinstance(stream, int) else stream.cuda_stream
    _check(lib().es_matrix_scan_static_f32(a.data_ptr(), sa, ra, b.data_ptr(), sb, rb, int(axis),
                                           int(bool(reverse)), int(bool(projective)), out.data_ptr(), handle))
    return out


def plan_linear_scan(a_shape, b_shape, axis: int = 0, reverse: bool = False,
                     ptrs: Optional[Sequence[int]] = None) -> dict:
    if ptrs is None:
        ptrs = [(k + 1) << 44 for k in range(3)]
    sa, ra = _shape_array(a_shape)
    sb, rb = _shape_array(b_shape)
    info = PlanInfo()
    _check(lib().es_plan_linear_scan_f32(ptrs[0], sa, ra, ptrs[1], sb, rb, int(axis), int(bool(reverse)), ptrs[2],
                                         ctypes.byref(info)))
    return _info(info)


def linear_scan(a, b, axis: int = 0, reverse: bool = False, out=None, stream=None):
    """linear-scan: h[t] = a[t] * h[t-1] + b[t] from h = 0, a and b broadcast
    to one shape (a Python number becomes a one-value device tensor)."""
    import torch
    dev = b.device if isinstance(b, torch.Tensor) else a.device
    if not isinstance(a, torch.Tensor):
        a = torch.tensor(float(a), device=dev, dtype=torch.float32)
    if not isinstance(b, torch.Tensor):
        b = torch.tensor(float(b), device=dev, dtype=torch.float32)
    _require_cuda_f32(a, "a")
    _require_cuda_f32(b, "b")
    shape = _lead_broadcast(list(a.shape), list(b.shape))
    if out is None:
        out = torch.empty(shape, device=dev, dtype=torch.float32)
    else:
        _require_cuda_f32(out, "out")
    sa, ra = _shape_array(a.shape)
    sb, rb = _shape_array(b.shape)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    handle = stream if isinstance(stream, int) else stream.cuda_stream
    _check(lib().es_linear_scan_f32(a.data_ptr(), sa, ra, b.data_ptr(), sb, rb, int(axis), int(bool(reverse)),
                                    out.data_ptr(), handle))
    return out


def plan_matrix_scan_backward(a_shape, b_shape, axis: int = 0, reverse: bool = False, projective: bool = False,
                              ptrs: Optional[Sequence[int]] = None) -> dict:
    """Validate and plan a matrix-scan backward without a GPU.  ``ptrs`` =
    (a, b, states, grad_out, grad_a, grad_b)."""
    if ptrs is None:
        ptrs = [(k + 1) << 44 for k in range(6)]
    sa, ra = _shape_array(a_shape)
    sb, rb = _shape_array(b_shape)
    info = PlanInfo()
    _check(lib().es_plan_matrix_scan_backward_f32(ptrs[0], sa, ra, ptrs[1], sb, rb, int(axis), int(bool(reverse)),
                                                  int(bool(projective)), ptrs[2], ptrs[3], ptrs[4], ptrs[5],
                                                  ctypes.byref(info)))
    return _info(info)


def _backward_args(a, b, states, grad_out, grads):
    import torch
    for t, nm in ((a, "a"), (b, "b"), (states, "states"), (grad_out, "grad_out")):
        _require_cuda_f32(t, nm)
    if list(grad_out.shape) != list(states.shape):
        raise EsError(1, "grad_out shape %s does not match the states %s" % (list(grad_out.shape),
                                                                             list(states.shape)))
    if grads is None:
        grads = (torch.empty_like(a), torch.empty_like(b))
    for t in grads:
        _require_cuda_f32(t, "gradient buffer")
    return grads


def matrix_scan_backward(a, b, states, grad_out, axis: int = 0, reverse: bool = False, projective: bool = False,
                         grads=None, stream=None):
    """Gradients (grad_a, grad_b) of sum(grad_out * matrix_scan(a, b)) on CUDA
    tensors, from the forward's states; ``grads`` may supply the buffers."""
    import torch
    ga, gb = _backward_args(a, b, states, grad_out, grads)
    sa, ra = _shape_array(a.shape)
    sb, rb = _shape_array(b.shape)
    if stream is None:
        stream = torch.cuda.current_stream(b.device)
    handle = stream if isinstance(stream, int) else stream.cuda_stream
    _check(lib().es_matrix_scan_backward_f32(a.data_ptr(), sa, ra, b.data_ptr(), sb, rb, int(axis),
                                             int(bool(reverse)), int(bool(projective)), states.data_ptr(),
                                             grad_out.data_ptr(), ga.data_ptr(), gb.data_ptr(), handle))
    return ga, gb


def plan_matrix_scan_backward_ws(a_shape, b_shape, workspace_bytes: int, axis: int = 0, reverse: bool = False,
                                 projective: bool = False, ptrs: Optional[Sequence[int]] = None) -> dict:
    """The checks and the kernel path of ``matrix_scan_backward_ws`` without a
    GPU.  ``ptrs`` = (a, b, states, grad_out, grad_a, grad_b, workspace)."""
    if ptrs is None:
        ptrs = [(k + 1) << 44 for k in range(7)]
    sa, ra = _shape_array(a_shape)
    sb, rb = _shape_array(b_shape)
    info = PlanInfo()
    _check(lib().es_plan_matrix_scan_backward_ws_f32(ptrs[0], sa, ra, ptrs[1], sb, rb, int(axis),
                                                     int(bool(reverse)), int(bool(projective)), ptrs[2], ptrs[3],
                                                     ptrs[4], ptrs[5], ptrs[6] if workspace_bytes else None,
                                                     int(workspace_bytes), ctypes.byref(info)))
    return _info(info)


def matrix_scan_backward_ws(a, b, states, grad_out, workspace, axis: int = 0, reverse: bool = False,
                            projective: bool = False, grads=None, stream=None):
    """matrix_scan_backward with a caller workspace (a CUDA tensor of at least
    ``matrix_scan_workspace`` bytes of the same shapes): few long lanes run the
    cotangent scan chunked."""
    import torch
    ga, gb = _backward_args(a, b, states, grad_out, grads)
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda:
        raise TypeError("workspace must be a CUDA tensor")
    sa, ra = _shape_array(a.shape)
    sb, rb = _shape_array(b.shape)
    if stream is None:
        stream = torch.cuda.current_stream(b.device)
    handle = stream if isinstance(stream, int) else stream.cuda_stream
    _check(lib().es_matrix_scan_backward_ws_f32(a.data_ptr(), sa, ra, b.data_ptr(), sb, rb, int(axis),
                                                int(bool(reverse)), int(bool(projective)), states.data_ptr(),
                                                grad_out.data_ptr(), ga.data_ptr(), gb.data_ptr(),
                                                workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                                handle))
    return ga, gb


def plan_linear_scan_backward(a_shape, b_shape, axis: int = 0, reverse: bool = False,
                              ptrs: Optional[Sequence[int]] = None) -> dict:
    if ptrs is None:
        ptrs = [(k + 1) << 44 for k in range(6)]
    sa, ra = _shape_array(a_shape)
    sb, rb = _shape_array(b_shape)
    info = PlanInfo()
    _check(lib().es_plan_linear_scan_backward_f32(ptrs[0], sa, ra, ptrs[1], sb, rb, int(axis), int(bool(reverse)),
                                                  ptrs[2], ptrs[3], ptrs[4], ptrs[5], ctypes.byref(info)))
    return _info(info)


def linear_scan_backward(a, b, states, grad_out, axis: int = 0, reverse: bool = False, grads=None, stream=None):
    """Gradients (grad_a, grad_b) of a linear-scan whose a and b share one shape."""
    import torch
    ga, gb = _backward_args(a, b, states, grad_out, grads)
    sa, ra = _shape_array(a.shape)
    sb, rb = _shape_array(b.shape)
    if stream is None:
        stream = torch.cuda.current_stream(b.device)
    handle = stream if isinstance(stream, int) else stream.cuda_stream
    _check(lib().es_linear_scan_backward_f32(a.data_ptr(), sa, ra, b.data_ptr(), sb, rb, int(axis),
                                             int(bool(reverse)), states.data_ptr(), grad_out.data_ptr(),
                                             ga.data_ptr(), gb.data_ptr(), handle))
    return ga, gb


# ---------------------------------------------------------------------------
# table-scan


def plan_table_scan(n_states: int, n_syms: int, shape, axis: int = -1, start: int = 0,
                    ptrs: Optional[Sequence[int]] = None) -> dict:
    """Validate and plan a table-scan without a GPU.  ``ptrs`` = (table,
    symbols, out), by default 16-byte aligned, non-overlapping stand-ins."""
    if ptrs is None:
        ptrs = [(k + 1) << 44 for k in range(3)]
    shp, rank = _shape_array(shape)
    info = PlanInfo()
    _check(lib().es_plan_table_scan_i32(ptrs[0], int(n_states), int(n_syms), ptrs[1], shp, rank, int(axis),
                                        int(start), ptrs[2], ctypes.byref(info)))
    return _info(info)


def table_scan(table, symbols, axis: int = -1, start: int = 0, out=None, stream=None):
    """table-scan on CUDA tensors: the automaton `table` ([states, symbols],
    int32) run over int32 `symbols` along `axis` from state `start`; returns
    the states (int32, `symbols`' shape)."""
    import torch
    for name, t in (("table", table), ("symbols", symbols)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
            raise TypeError("%s must be a contiguous CUDA tensor" % name)
        if t.dtype != torch.int32:
            raise EsError(2, "E-DIM-002 table-scan: %s is %s; table and symbols must be i32" % (name, t.dtype))
    if table.dim() != 2:
        raise EsError(1, "E-DIM-001 table-scan: the table must be [states symbols], got rank %d" % table.dim())
    if out is None:
        out = torch.empty(symbols.shape, device=symbols.device, dtype=torch.int32)
    shp, rank = _shape_array(symbols.shape)
    if stream is None:
        stream = torch.cuda.current_stream(symbols.device)
    handle = stream if isinstance(stream, int) else stream.cuda_stream
    _check(lib().es_table_scan_i32(table.data_ptr(), int(table.shape[0]), int(table.shape[1]), symbols.data_ptr(),
                                   shp, rank, int(axis), int(start), out.data_ptr(), handle))
    return out
