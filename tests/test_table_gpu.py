"""table-scan on the GPU against the oracle, bit for bit (integer work), on
every kernel: time innermost, sequences side by side, generic; tables in
shared memory and in global memory; clamping of symbols and entries; the
pages' parity example."""
import json
import os

import numpy as np
import pytest
import torch

import oracle.table as TS
from element_scan_recurrences_gb300 import binding as es

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    es.lib()
    yield
    es.set_path_override("auto")


def run(table, sym, axis=-1, start=0, path="auto", expect=None):
    es.set_path_override(path)
    try:
        if expect is not None:
            assert es.plan_table_scan(table.shape[0], table.shape[1], sym.shape, axis, start)["path"] == expect
        got = es.table_scan(torch.from_numpy(table).cuda(), torch.from_numpy(sym).cuda(), axis=axis, start=start)
        es.device_status()
        return got.cpu().numpy()
    finally:
        es.set_path_override("auto")


def random_table(rng, states, syms, lo=None, hi=None):
    lo = 0 if lo is None else lo
    hi = states if hi is None else hi
    return rng.integers(lo, hi, (states, syms)).astype(np.int32)


def test_parity_example():
    g = json.load(open(os.path.join(GOLDEN, "table_scan_parity.json")))
    got = run(np.array(g["table"], np.int32), np.array(g["symbols"], np.int32))
    assert np.array_equal(got, np.array(g["expected"], np.int32))


@pytest.mark.parametrize("states,syms", [(2, 2), (64, 16), (300, 100), (4096, 16)],
                         ids=["tiny", "small", "medium", "large_table_in_global"])
def test_time_innermost(states, syms):
    rng = np.random.default_rng(states)
    table = random_table(rng, states, syms)
    sym = rng.integers(0, syms, (150, 100)).astype(np.int32)     # a ragged row tile and trip tile
    for start in (0, states - 1):
        got = run(table, sym, -1, start, expect="time_tma")
        assert np.array_equal(got, TS.table_scan(table, sym, -1, start))
        got = run(table, sym, -1, start, path="generic")
        assert np.array_equal(got, TS.table_scan(table, sym, -1, start))


@pytest.mark.parametrize("states,syms", [(5, 3), (64, 16), (4096, 16)])
def test_sequences_side_by_side(states, syms):
    rng = np.random.default_rng(states + 1)
    table = random_table(rng, states, syms)
    sym = rng.integers(0, syms, (3, 70, 200)).astype(np.int32)
    got = run(table, sym, 1, 1 % states, expect="lane_tma")
    assert np.array_equal(got, TS.table_scan(table, sym, 1, 1 % states))
    got = run(table, sym, 0, 0, path="generic")
    assert np.array_equal(got, TS.table_scan(table, sym, 0, 0))


def test_clamping_on_every_path():
    rng = np.random.default_rng(9)
    states, syms = 40, 8
    table = random_table(rng, states, syms, lo=-10, hi=states + 10)     # entries out of range
    sym = rng.integers(-3, syms + 3, (130, 64)).astype(np.int32)           # symbols out of range
    want = TS.table_scan(table, sym)
    assert np.array_equal(run(table, sym, expect="time_tma"), want)
    assert np.array_equal(run(table, sym, path="generic"), want)
    sym3 = rng.integers(-3, syms + 3, (2, 64, 132)).astype(np.int32)
    assert np.array_equal(run(table, sym3, 1, expect="lane_tma"), TS.table_scan(table, sym3, 1))
    got = run(table, sym3, 1)
    assert got.min() >= 0 and got.max() < states


@pytest.mark.parametrize("name", ["table_scan_time_inner", "table_scan_lanes"])
def test_full_size_every_element(name):
    """The bench workloads at full size, every state against the oracle (run
    on every host core over contiguous blocks of rows), bit for bit."""
    import oracle
    from element_scan_recurrences_gb300 import workloads as wl
    w = wl.TABLE_WORKLOADS[name]
    table, sym = wl.make_table_inputs(w, "cuda")
    out = es.table_scan(table, sym, axis=w.axis)
    es.device_status()
    th, sh = table.cpu().numpy(), sym.cpu().numpy()
    want = np.empty(tuple(out.shape), np.int32)

    def rows(lo, hi):
        want[lo:hi] = TS.table_scan(th, sh[lo:hi], axis=w.axis)
    oracle.split_rows(rows, w.shape[0])
    assert np.array_equal(out.cpu().numpy(), want)
