"""CPU oracle for `table-scan` -- TEST INFRASTRUCTURE.

Like the rest of this package, only the test suite, ``__graft_entry__.smoke()``
and the bench's CPU-baseline and reference arms may import it; it shares no
code with the CUDA library.

What it computes ("Tensor operations": the `table-scan` row of the operations
table and the section "table-scan"): a deterministic automaton run along
`axis` of `symbols` (the last by default),

    h[t] = table[h[t-1], symbols[t]]      from h[-1] = start (0 by default),

the result holding every state, in `symbols`' shape; `table` is
[states, symbols], both tensors i32.  On CUDA a symbol outside [0, symbols)
and a table entry the run reaches outside [0, states) are clamped into range
(as `gather` clamps an index there); the CPU and Metal backends refuse them.
Reading: the clamped entry is the state, so every stored state lies in
[0, states).  Shape errors are E-DIM-001 (a table that is not rank 2 or has
no symbols, an axis out of range, a start that is not a state); dtypes other
than i32 are E-DIM-002.
"""
from __future__ import annotations

import numpy as np

__all__ = ["table_scan", "TableScanError"]


class TableScanError(ValueError):
    def __init__(self, code, msg):
        super().__init__("%s: %s" % (code, msg))
        self.code = code


def table_scan(table, symbols, axis=-1, start=0, clamp=True):
    """Run the automaton; ``clamp=False`` refuses out-of-range symbols and
    entries as the CPU backend does (raises TableScanError)."""
    table = np.asarray(table)
    symbols = np.asarray(symbols)
    if table.dtype != np.int32 or symbols.dtype != np.int32:
        raise TableScanError("E-DIM-002", "table and symbols must be i32")
    if table.ndim != 2 or table.shape[1] == 0 or table.shape[0] == 0:
        raise TableScanError("E-DIM-001", "table must be [states symbols] with at least one of each")
    if symbols.ndim == 0:
        raise TableScanError("E-DIM-001", "symbols need an axis")
    ax = axis + symbols.ndim if axis < 0 else axis
    if not 0 <= ax < symbols.ndim:
        raise TableScanError("E-DIM-001", "axis %d out of range" % axis)
    n_states, n_syms = table.shape
    if not 0 <= start < n_states:
        raise TableScanError("E-DIM-001", "start %d is not a state" % start)
    sym = np.moveaxis(symbols, ax, -1)
    lanes_shape = sym.shape[:-1]
    T = sym.shape[-1]
    sym = sym.reshape(-1, T)
    h = np.full(sym.shape[0], start, dtype=np.int64)
    out = np.empty(sym.shape, dtype=np.int32)
    for t in range(T):
        s = sym[:, t].astype(np.int64)
        if clamp:
            s = np.clip(s, 0, n_syms - 1)
        elif np.any((s < 0) | (s >= n_syms)):
            raise TableScanError("E-RANGE", "a symbol outside [0, %d)" % n_syms)
        nxt = table[h, s].astype(np.int64)
        if clamp:
            nxt = np.clip(nxt, 0, n_states - 1)
        elif np.any((nxt < 0) | (nxt >= n_states)):
            raise TableScanError("E-RANGE", "a table entry outside [0, %d)" % n_states)
        h = nxt
        out[:, t] = h
    return np.moveaxis(out.reshape(lanes_shape + (T,)), -1, ax)
