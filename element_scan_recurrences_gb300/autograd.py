"""Differentiable element scans for PyTorch graphs.

``element_scan(body, initial, sequences, ...)`` runs the forward scan through
the C ABI and registers its backward ("Nonlinear element scans", "Precision
and gradients": gradients flow to `initial` and every sequence; the gradient
is another element scan in the opposite trip order applying the body's
vector-Jacobian product over the saved states).  This module only marshals
arguments between autograd and the library: both passes run in the CUDA
kernels, and CPU tensors are refused (no fallback).

``matrix_scan(a, b, ...)`` and ``linear_scan(a, b, ...)`` are differentiable
the same way ("matrix-scan": the gradient is the same scan run backwards on
a's transposes; a projective scan has none, and its backward raises).

A parameter shared along time or lanes is broadcast to the sequence shape
before the call, as the pages ask ("Arguments and body": parameters enter
through the sequence list).  Done with ``expand`` (then made contiguous for
the kernels), autograd sums the parameter's gradient over time and the other
broadcast axes; a tensor passed as two sequences, or read again elsewhere,
accumulates its gradients the same way.  The backward itself is not
differentiated again.
"""
from __future__ import annotations

import threading
from typing import Sequence

import torch
from torch.autograd.function import once_differentiable

from . import binding as es

_programs = {}
_programs_lock = threading.Lock()


def _program(text: str) -> "es.Body":
    """One compiled program per body text (kernels are cached by the library)."""
    with _programs_lock:
        b = _programs.get(text)
        if b is None:
            b = _programs[text] = es.Body(text)
        return b


class _Scan(torch.autograd.Function):
    @staticmethod
    def forward(ctx, body, axis, state_axis, reverse, initial, *seqs):
        if isinstance(body, es.Body):
            out = body.scan(initial, list(seqs), axis=axis, state_axis=state_axis, reverse=reverse)
        else:
            out = es.scan(body, initial, list(seqs), axis=axis, state_axis=state_axis, reverse=reverse)
        ctx.body, ctx.axis, ctx.state_axis, ctx.reverse = body, axis, state_axis, reverse
        ctx.save_for_backward(initial, out, *seqs)
        return out

    @staticmethod
    @once_differentiable
    def backward(ctx, grad_out):
        initial, out, *seqs = ctx.saved_tensors
        grad_out = grad_out.contiguous()
        if isinstance(ctx.body, es.Body):
            gi, gs = ctx.body.scan_backward(initial, seqs, out, grad_out, axis=ctx.axis, state_axis=ctx.state_axis,
                                            reverse=ctx.reverse)
        else:
            gi, gs = es.scan_backward(ctx.body, initial, seqs, out, grad_out, axis=ctx.axis,
                                      state_axis=ctx.state_axis, reverse=ctx.reverse)
        return (None, None, None, None, gi) + tuple(gs)


def element_scan(body, initial: torch.Tensor, sequences: Sequence[torch.Tensor], axis: int = 0,
                 state_axis: bool = False, reverse: bool = False) -> torch.Tensor:
    """The states of an element scan, differentiable with respect to
    `initial` and every sequence.

    ``body`` is a body program's text, an ``es.Body``, or one of the
    built-in bodies (``es.TANH_DECAY``, ``es.NORMCAP``, ``es.MAXPLUS`` or
    their names).  Tensors are CUDA float32; non-contiguous ones are copied
    to contiguous ones first.
    """
    if isinstance(body, str) and body.lstrip().startswith("("):
        body = _program(body)
    seqs = [s.contiguous() for s in sequences]
    return _Scan.apply(body, int(axis), bool(state_axis), bool(reverse), initial.contiguous(), *seqs)


class _MatrixScan(torch.autograd.Function):
    @staticmethod
    def forward(ctx, linear, axis, reverse, projective, chunked, a, b):
        ws = None
        if chunked and not linear:
            nbytes = es.matrix_scan_workspace(a.shape, b.shape, axis, projective)
            if nbytes:
                ws = torch.empty(nbytes, dtype=torch.uint8, device=a.device)
        if linear:
            out = es.linear_scan(a, b, axis=axis, reverse=reverse)
        elif ws is not None:
            out = es.matrix_scan_ws(a, b, ws, axis=axis, reverse=reverse, projective=projective)
        else:
            out = es.matrix_scan(a, b, axis=axis, reverse=reverse, projective=projective)
        ctx.linear, ctx.axis, ctx.reverse, ctx.projective, ctx.ws = linear, axis, reverse, projective, ws
        ctx.save_for_backward(a, b, out)
        return out

    @staticmethod
    @once_differentiable
    def backward(ctx, grad_out):
        a, b, out = ctx.saved_tensors
        grad_out = grad_out.contiguous()
        if ctx.linear:
            ga, gb = es.linear_scan_backward(a, b, out, grad_out, axis=ctx.axis, reverse=ctx.reverse)
        elif ctx.ws is not None:
            ga, gb = es.matrix_scan_backward_ws(a, b, out, grad_out, ctx.ws, axis=ctx.axis, reverse=ctx.reverse,
                                                projective=ctx.projective)
        else:
            ga, gb = es.matrix_scan_backward(a, b, out, grad_out, axis=ctx.axis, reverse=ctx.reverse,
                                             projective=ctx.projective)
        return None, None, None, None, None, ga, gb


def _one_shape(a, b, lead_a, lead_b):
    """Broadcast the leading dims of a and b to one shape (autograd sums a
    broadcast operand's gradient back)."""
    r = max(len(lead_a), len(lead_b))
    la = [1] * (r - len(lead_a)) + list(lead_a)
    lb = [1] * (r - len(lead_b)) + list(lead_b)
    lead = [y if x == 1 else x for x, y in zip(la, lb)]
    a = a.reshape(la + list(a.shape[len(lead_a):])).expand(lead + list(a.shape[len(lead_a):]))
    b = b.reshape(lb + list(b.shape[len(lead_b):])).expand(lead + list(b.shape[len(lead_b):]))
    return a.contiguous(), b.contiguous()


def matrix_scan(a: torch.Tensor, b: torch.Tensor, axis: int = 0, reverse: bool = False,
                projective: bool = False, chunked: bool = False) -> torch.Tensor:
    """The states of a matrix-scan, differentiable with respect to a and b
    (leading dims broadcast first, so autograd sums a shared operand's
    gradient).  ``chunked``: few long lanes run the chunked scan and the
    chunked gradient in a workspace allocated here (results within rounding
    of the sequential scan, not bit for bit); other shapes are unaffected."""
    a, b = _one_shape(a, b, a.shape[:-2], b.shape[:-2])
    return _MatrixScan.apply(False, int(axis), bool(reverse), bool(projective), bool(chunked), a, b)


def linear_scan(a: torch.Tensor, b: torch.Tensor, axis: int = 0, reverse: bool = False) -> torch.Tensor:
    """The states of a linear-scan, differentiable with respect to a and b."""
    a, b = _one_shape(a, b, a.shape, b.shape)
    return _MatrixScan.apply(True, int(axis), bool(reverse), False, False, a, b)
