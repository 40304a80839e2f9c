"""Differentiable element scans for PyTorch graphs.

``element_scan(body, initial, sequences, ...)`` runs the forward scan through
the C ABI and registers its backward ("Nonlinear element scans", "Precision
and gradients": gradients flow to `initial` and every sequence; the gradient
is another element scan in the opposite trip order applying the body's
vector-Jacobian product over the saved states).  This module only marshals
arguments between autograd and the library: both passes run in the CUDA
kernels, and CPU tensors are refused (no fallback).

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
