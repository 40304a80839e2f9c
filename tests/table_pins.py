"""Pins of the table-scan oracle (``oracle.table``) to facts from outside it.

  * the pages' worked example: the parity automaton [[0 1] [1 0]] gives the
    parity so far (golden fixture, hand-derived);
  * a counter modulo k (table[h, s] = (h + s) mod k) is the running sum mod k
    (``np.cumsum``); a shift register (table[h, s] = (2h + s) mod 2^w) holds
    the last w symbols, read straight off the input;
  * a start state offsets the counter; the axis may sit anywhere;
  * CUDA's clamping: symbols below 0 act as 0 and above the alphabet as its
    last symbol; table entries are clamped into [0, states); the refusing
    (CPU backend) mode raises instead;
  * shapes and dtypes the contract rejects.
"""
from __future__ import annotations

import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
i32 = np.int32


def pin_parity_example(T):
    g = json.load(open(os.path.join(GOLDEN, "table_scan_parity.json")))
    got = T.table_scan(np.array(g["table"], i32), np.array(g["symbols"], i32), axis=g["axis"], start=g["start"])
    assert np.array_equal(got, np.array(g["expected"], i32)), got


def pin_counter_and_shift_register(T):
    rng = np.random.default_rng(1)
    k = 7
    table = ((np.arange(k)[:, None] + np.arange(5)[None, :]) % k).astype(i32)      # 5 symbols
    sym = rng.integers(0, 5, (3, 40)).astype(i32)
    assert np.array_equal(T.table_scan(table, sym), (np.cumsum(sym, axis=1) % k).astype(i32)), "counter"
    assert np.array_equal(T.table_scan(table, sym, start=3), ((3 + np.cumsum(sym, axis=1)) % k).astype(i32)), \
        "start state"
    # shift register of the last 3 bits
    w = 3
    table = ((2 * np.arange(2 ** w)[:, None] + np.arange(2)[None, :]) % (2 ** w)).astype(i32)
    bits = rng.integers(0, 2, (4, 30)).astype(i32)
    got = T.table_scan(table, bits)
    want = np.zeros_like(bits)
    for d in range(w):
        want[:, d:] += bits[:, :bits.shape[1] - d] << d
    assert np.array_equal(got, want), "shift register"
    # the axis elsewhere: the same run on the transposed layout
    got0 = T.table_scan(table, np.ascontiguousarray(bits.T), axis=0)
    assert np.array_equal(got0, want.T), "axis 0"


def pin_clamping(T):
    table = np.array([[1, 2, 0], [2, 0, 1], [0, 1, 2]], i32)
    # symbols out of range act as the nearest symbol
    sym = np.array([[-5, 7, 1, 99, -1]], i32)
    want = T.table_scan(table, np.clip(sym, 0, 2).astype(i32))
    assert np.array_equal(T.table_scan(table, sym), want), "symbol clamp"
    # table entries out of range are clamped into [0, states)
    bad = np.array([[5, -3], [1, 9]], i32)
    got = T.table_scan(bad, np.array([[0, 1, 0, 1]], i32))
    # h: start 0 -> bad[0,0]=5->1 -> bad[1,1]=9->1 -> bad[1,0]=1 -> bad[1,1]=9->1
    assert np.array_equal(got, np.array([[1, 1, 1, 1]], i32)), got
    assert np.array_equal(T.table_scan(bad, np.array([[1, 0]], i32)), np.array([[0, 1]], i32))
    for sy, tb in ((sym, table), (np.array([[0, 1]], i32), bad)):
        try:
            T.table_scan(tb, sy, clamp=False)
        except ValueError:
            continue
        raise AssertionError("the refusing mode accepted an out-of-range run")


def pin_rejected(T):
    ok_table = np.zeros((2, 2), i32)
    cases = [
        (np.zeros((2, 2), np.float32), np.zeros((1, 3), i32), -1, 0),   # dtype
        (ok_table, np.zeros((1, 3), np.int64), -1, 0),                   # dtype
        (np.zeros((2,), i32), np.zeros((1, 3), i32), -1, 0),             # table rank
        (np.zeros((2, 0), i32), np.zeros((1, 3), i32), -1, 0),           # no symbols
        (ok_table, np.zeros((1, 3), i32), 2, 0),                         # axis out of range
        (ok_table, np.zeros((1, 3), i32), -1, 2),                        # start not a state
        (ok_table, np.zeros((1, 3), i32), -1, -1),                       # start not a state
    ]
    for table, sym, axis, start in cases:
        try:
            T.table_scan(table, sym, axis=axis, start=start)
        except ValueError:
            continue
        raise AssertionError("accepted a call the contract rejects")


ALL_PINS = [pin_parity_example, pin_counter_and_shift_register, pin_clamping, pin_rejected]
