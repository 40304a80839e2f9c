"""Seeded synthetic inputs for `element-scan` workloads.

This module only draws random numbers and describes shapes: it holds none of
the scan's arithmetic, so both the CUDA path and the CPU oracle may be fed
from it.  Every draw comes from one ``torch.Generator`` seeded per workload,
in the order x, then the second sequence (decay / gate / cost), then initial.

Distributions: ``("normal", mu, sigma)`` is ``mu + sigma * randn``;
``("uniform", lo, hi)`` is ``lo + (hi - lo) * rand``; ``("const", v)`` is a
constant fill.  The five named workloads are the element-scan cases the
library is measured and checked on: a small TANH_DECAY case, a wide-lane
TANH_DECAY case, a NORMCAP vector-state case, a reverse MAXPLUS case and a
TANH_DECAY case whose sequence axis is innermost.  The ``body_*`` workloads
run body programs (the body given as text) on the same shapes: the pages'
bodies, to set the run-time compiled kernels beside the built-in ones, and a
gated body with three sequences.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import torch

TANH_DECAY = 0
NORMCAP = 1
MAXPLUS = 2
BODY_PROGRAM = -1
BODY_NAMES = {TANH_DECAY: "TANH_DECAY", NORMCAP: "NORMCAP", MAXPLUS: "MAXPLUS", BODY_PROGRAM: "program"}

# the pages' bodies as text ("Nonlinear element scans": intro, :state-axis
# and :reverse examples) and a gated variant with a third sequence
TANH_DECAY_TEXT = "(lambda (h x a) (tanh (+ x (* a h))))"
NORMCAP_TEXT = ("(lambda (h x a) (let ((y (+ (* a h) x))) "
                "(/ y (maximum 1.0 (sqrt (sum (* y y) :axes [-1]))))))")
MAXPLUS_TEXT = "(lambda (h x c) (maximum (- h c) x))"
GATED_TEXT = "(lambda (h x a g) (where (> g 0.5) (tanh (+ x (* a h))) h))"


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    body: int
    shape: Tuple[int, ...]            # output shape (= full-width sequence shape)
    axis: int
    state_axis: bool
    seq_widths: Tuple[int, int]       # last width of x and of the second sequence
    reverse: Tuple[bool, ...]         # directions that are run
    x_dist: tuple
    a_dist: tuple
    init_dist: tuple
    seed: int = 0
    text: Optional[str] = None        # a body program (then `body` is BODY_PROGRAM)
    extra_dists: tuple = ()           # distributions of sequences after the second

    @property
    def n_seqs(self) -> int:
        return 2 + len(self.extra_dists)

    @property
    def rank(self) -> int:
        return len(self.shape)

    @property
    def ax(self) -> int:
        return self.axis + self.rank if self.axis < 0 else self.axis

    @property
    def T(self) -> int:
        return self.shape[self.ax]

    @property
    def elements(self) -> int:
        return math.prod(self.shape)

    def seq_shape(self, k: int) -> Tuple[int, ...]:
        s = list(self.shape)
        if self.state_axis:
            s[-1] = self.seq_widths[k]
        return tuple(s)

    @property
    def init_shape(self) -> Tuple[int, ...]:
        return tuple(d for i, d in enumerate(self.shape) if i != self.ax)

    def algorithmic_bytes(self) -> int:
        """f32 bytes read (every sequence and initial) plus states written."""
        reads = sum(math.prod(self.seq_shape(k)) for k in range(self.n_seqs))
        return 4 * (reads + math.prod(self.init_shape) + self.elements)

    def backward_algorithmic_bytes(self, live_mask: Optional[int] = None) -> int:
        """f32 bytes of one backward launch: the output gradient, the saved
        states, the second sequence, x (not for TANH_DECAY, whose gradient
        never reads it) and initial read; both sequence gradients and the
        initial gradient written.  A body program's backward reads the
        sequences its vector-Jacobian product reads (bit k of `live_mask`;
        all when None) and writes every sequence's gradient."""
        ni = math.prod(self.init_shape)
        if self.text is not None:
            sizes = [math.prod(self.seq_shape(k)) for k in range(self.n_seqs)]
            live = sum(n for k, n in enumerate(sizes) if live_mask is None or (live_mask >> k) & 1)
            return 4 * (2 * self.elements + live + ni + sum(sizes) + ni)
        n0, n1 = (math.prod(self.seq_shape(k)) for k in range(2))
        reads = 2 * self.elements + n1 + ni + (0 if self.body == TANH_DECAY else n0)
        return 4 * (reads + n0 + n1 + ni)

    def with_shape(self, shape: Sequence[int], name: Optional[str] = None) -> "Workload":
        """Same body, axis and distributions at another shape."""
        return dataclasses.replace(self, shape=tuple(shape), name=name or self.name + "@" + "x".join(map(str, shape)))


WORKLOADS = {
    w.name: w for w in [
        Workload("tanh_decay_small", TANH_DECAY, (2, 64, 8), 1, False, (8, 8), (False,),
                 ("normal", 0.0, 1.0), ("uniform", 0.0, 0.9), ("normal", 0.0, 0.1)),
        Workload("tanh_decay_lanes", TANH_DECAY, (64, 4096, 1024), 1, False, (1024, 1024), (False,),
                 ("normal", 0.0, 1.0), ("uniform", 0.5, 0.99), ("const", 0.0)),
        Workload("normcap_vector", NORMCAP, (32, 8192, 64, 16), 1, True, (16, 1), (False,),
                 ("normal", 0.0, 0.5), ("uniform", 0.8, 1.0), ("const", 0.0)),
        Workload("maxplus_reverse", MAXPLUS, (128, 16384, 128), 1, False, (128, 128), (True,),
                 ("uniform", -1.0, 1.0), ("uniform", 0.0, 0.1), ("const", -3.0e38)),
        Workload("tanh_decay_time_inner", TANH_DECAY, (262144, 1024), -1, False, (1024, 1024), (False, True),
                 ("normal", 0.0, 1.0), ("uniform", 0.5, 0.99), ("normal", 0.0, 0.1)),
        Workload("body_tanh_decay_lanes", BODY_PROGRAM, (64, 4096, 1024), 1, False, (1024, 1024), (False,),
                 ("normal", 0.0, 1.0), ("uniform", 0.5, 0.99), ("const", 0.0), text=TANH_DECAY_TEXT),
        Workload("body_gated_lanes", BODY_PROGRAM, (64, 4096, 1024), 1, False, (1024, 1024, 1024), (False,),
                 ("normal", 0.0, 1.0), ("uniform", 0.5, 0.99), ("const", 0.0), text=GATED_TEXT,
                 extra_dists=(("uniform", 0.0, 1.0),)),
        Workload("body_normcap_vector", BODY_PROGRAM, (32, 8192, 64, 16), 1, True, (16, 1), (False,),
                 ("normal", 0.0, 0.5), ("uniform", 0.8, 1.0), ("const", 0.0), text=NORMCAP_TEXT),
        Workload("body_maxplus_reverse", BODY_PROGRAM, (128, 16384, 128), 1, False, (128, 128), (True,),
                 ("uniform", -1.0, 1.0), ("uniform", 0.0, 0.1), ("const", -3.0e38), text=MAXPLUS_TEXT),
        Workload("body_tanh_decay_time_inner", BODY_PROGRAM, (262144, 1024), -1, False, (1024, 1024),
                 (False, True), ("normal", 0.0, 1.0), ("uniform", 0.5, 0.99), ("normal", 0.0, 0.1),
                 text=TANH_DECAY_TEXT),
    ]
}
ORDER = ["tanh_decay_small", "tanh_decay_lanes", "normcap_vector", "maxplus_reverse",
         "tanh_decay_time_inner"]
BODY_ORDER = ["body_tanh_decay_lanes", "body_gated_lanes", "body_normcap_vector", "body_maxplus_reverse",
              "body_tanh_decay_time_inner"]


def _draw(dist: tuple, shape, gen: torch.Generator, device) -> torch.Tensor:
    kind = dist[0]
    if kind == "normal":
        t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        return t.mul_(dist[2]).add_(dist[1])
    if kind == "uniform":
        t = torch.rand(shape, generator=gen, device=device, dtype=torch.float32)
        return t.mul_(dist[2] - dist[1]).add_(dist[1])
    if kind == "const":
        return torch.full(shape, dist[1], device=device, dtype=torch.float32)
    raise ValueError("unknown distribution %r" % (dist,))


def make_inputs(w: Workload, device="cpu", seed: Optional[int] = None):
    """Draw (initial, [x, second, ...]) for a workload, seeded, on ``device``:
    the sequences in order, then initial."""
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    dists = (w.x_dist, w.a_dist) + tuple(w.extra_dists)
    seqs = [_draw(d, w.seq_shape(k), gen, device) for k, d in enumerate(dists)]
    init = _draw(w.init_dist, w.init_shape, gen, device)
    return init, seqs


def custom(body: int, shape, axis: int, state_axis: bool = False, seq_widths=None,
           reverse: bool = False, x_dist=("normal", 0.0, 1.0), a_dist=("uniform", 0.5, 0.99),
           init_dist=("normal", 0.0, 0.1), seed: int = 0, name: str = "custom") -> Workload:
    """An ad-hoc workload (tests use it for shapes outside the named five)."""
    shape = tuple(int(d) for d in shape)
    if seq_widths is None:
        seq_widths = (shape[-1], shape[-1])
    return Workload(name, body, shape, axis, state_axis, tuple(seq_widths), (reverse,),
                    x_dist, a_dist, init_dist, seed)


# ---------------------------------------------------------------------------
# matrix-scan / linear-scan workloads ("Tensor operations", section
# "matrix-scan": the delta rule S[t] = (I - beta k k^T) S[t-1] + beta k v^T
# over [b t n m]; linear-scan over one-by-one matrices)


@dataclasses.dataclass(frozen=True)
class MatrixWorkload:
    name: str
    kind: str                      # "delta_rule" (matrix-scan) or "linear" (linear-scan)
    lead: Tuple[int, ...]          # leading shape; the scanned axis is `axis`
    axis: int
    n: int
    m: int
    reverse: Tuple[bool, ...] = (False,)
    projective: bool = False
    seed: int = 0
    workspace: bool = False        # run through the workspace entry (chunked scan for few lanes)

    @property
    def ax(self) -> int:
        return self.axis + len(self.lead) if self.axis < 0 else self.axis

    @property
    def T(self) -> int:
        return self.lead[self.ax]

    @property
    def a_shape(self) -> Tuple[int, ...]:
        return self.lead + ((self.n, self.n) if self.kind != "linear" else ())

    @property
    def b_shape(self) -> Tuple[int, ...]:
        return self.lead + ((self.n, self.m) if self.kind != "linear" else ())

    @property
    def shape(self) -> Tuple[int, ...]:
        return self.b_shape

    @property
    def elements(self) -> int:
        return math.prod(self.b_shape)

    def algorithmic_bytes(self) -> int:
        """f32 bytes of one launch: a and b read, the states written."""
        return 4 * (math.prod(self.a_shape) + 2 * math.prod(self.b_shape))

    def backward_algorithmic_bytes(self) -> int:
        """f32 bytes of one backward call: a, the saved states and the state
        gradients read; the gradients of a and of b written."""
        na, nb = math.prod(self.a_shape), math.prod(self.b_shape)
        return 4 * (2 * na + 3 * nb)

    def with_trips(self, T: int, name: Optional[str] = None) -> "MatrixWorkload":
        lead = tuple(T if i == self.ax else d for i, d in enumerate(self.lead))
        return dataclasses.replace(self, lead=lead, name=name or "%s_T%d" % (self.name, T))


MATRIX_WORKLOADS = {
    w.name: w for w in [
        # the pages' delta rule: 64 sequences x 16 heads, 1024 steps, 16 x 16 state
        MatrixWorkload("matrix_scan_delta_rule", "delta_rule", (64, 1024, 16), 1, 16, 16),
        # the delta rule over 8 long sequences: few lanes, run as a chunked scan
        MatrixWorkload("matrix_scan_few_lanes", "delta_rule", (8, 131072), 1, 16, 16, workspace=True),
        # linear-scan on the shape of the wide-lane element-scan case
        MatrixWorkload("linear_scan_lanes", "linear", (64, 4096, 1024), 1, 1, 1),
    ]
}


def make_matrix_inputs(w: MatrixWorkload, device="cpu", seed: Optional[int] = None):
    """Draw (a, b) for a matrix workload, seeded, on ``device``.

    delta_rule: keys k ~ N(0, 1) normalised to unit length, values
    v ~ N(0, 1), beta ~ U(0, 1), drawn in that order; a = I - beta k k^T and
    b = beta k v^T are formed from them (input construction: outer products of
    the drawn vectors).  linear: a ~ U(0.5, 0.99), then b ~ N(0, 1)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    if w.kind == "linear":
        a = torch.rand(w.lead, generator=gen, device=device).mul_(0.49).add_(0.5)
        b = torch.randn(w.lead, generator=gen, device=device)
        return a, b
    k = torch.randn(w.lead + (w.n,), generator=gen, device=device)
    k = k / k.norm(dim=-1, keepdim=True)
    v = torch.randn(w.lead + (w.m,), generator=gen, device=device)
    beta = torch.rand(w.lead + (1, 1), generator=gen, device=device)
    eye = torch.eye(w.n, device=device)
    a = (eye - beta * k.unsqueeze(-1) * k.unsqueeze(-2)).contiguous()
    b = (beta * k.unsqueeze(-1) * v.unsqueeze(-2)).contiguous()
    return a, b


# ---------------------------------------------------------------------------
# table-scan workloads ("Tensor operations", section "table-scan"): a random
# automaton over random symbols


@dataclasses.dataclass(frozen=True)
class TableWorkload:
    name: str
    shape: Tuple[int, ...]         # symbols' shape
    axis: int
    n_states: int
    n_syms: int
    seed: int = 0
    reverse: Tuple[bool, ...] = (False,)   # table-scan runs forward only

    @property
    def ax(self) -> int:
        return self.axis + len(self.shape) if self.axis < 0 else self.axis

    @property
    def T(self) -> int:
        return self.shape[self.ax]

    @property
    def elements(self) -> int:
        return math.prod(self.shape)

    def algorithmic_bytes(self) -> int:
        """i32 bytes of one launch: symbols read, states written, the table."""
        return 4 * (2 * self.elements + self.n_states * self.n_syms)

    def with_trips(self, T: int, name: Optional[str] = None) -> "TableWorkload":
        shape = tuple(T if i == self.ax else d for i, d in enumerate(self.shape))
        return dataclasses.replace(self, shape=shape, name=name or "%s_T%d" % (self.name, T))


TABLE_WORKLOADS = {
    w.name: w for w in [
        # sequences as rows, the pages' default axis (the last)
        TableWorkload("table_scan_time_inner", (262144, 1024), -1, 64, 16),
        # sequences side by side
        TableWorkload("table_scan_lanes", (64, 4096, 1024), 1, 64, 16),
    ]
}


def make_table_inputs(w: TableWorkload, device="cpu", seed: Optional[int] = None):
    """(table, symbols), seeded: table entries uniform in [0, states), then
    symbols uniform in [0, symbols); both int32."""
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    table = torch.randint(0, w.n_states, (w.n_states, w.n_syms), generator=gen, device=device, dtype=torch.int32)
    sym = torch.randint(0, w.n_syms, w.shape, generator=gen, device=device, dtype=torch.int32)
    return table, sym
