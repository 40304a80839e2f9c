"""The all-cores oracle (lanes split into contiguous blocks along dim 0, each
block scanned by the unchanged single-thread loop) gives the single-thread
result bit for bit, forward and backward, on ragged splits, with and without
a state axis and with the sequence axis innermost."""
import numpy as np
import pytest

import oracle

CASES = [
    # body, shape, axis, state_axis, seq_widths
    (oracle.TANH_DECAY, (7, 33, 5), 1, False, None),
    (oracle.MAXPLUS, (11, 3, 40), 1, False, None),
    (oracle.TANH_DECAY, (13, 29), -1, False, None),
    (oracle.NORMCAP, (5, 17, 3, 16), 1, True, (16, 1)),
    (oracle.NORMCAP, (6, 9, 2, 4), 1, True, (4, 4)),
    (oracle.TANH_DECAY, (3, 4, 10, 6), 2, False, None),
]


def _inputs(body, shape, axis, state_axis, widths, seed):
    rng = np.random.default_rng(seed)
    rank = len(shape)
    ax = axis % rank
    sh = [list(shape), list(shape)]
    if state_axis:
        sh[0][-1], sh[1][-1] = widths
    x = rng.standard_normal(sh[0]).astype(np.float32)
    if body == oracle.MAXPLUS:
        a = rng.uniform(0.0, 0.1, sh[1]).astype(np.float32)
    else:
        a = rng.uniform(0.5, 0.99, sh[1]).astype(np.float32)
    init = rng.standard_normal([d for i, d in enumerate(shape) if i != ax]).astype(np.float32) * 0.1
    return init, [x, a]


@pytest.mark.parametrize("threads", [2, 3, 64])
@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[1])))
def test_threaded_oracle_is_bit_identical(case, reverse, threads):
    body, shape, axis, sa, widths = case
    init, seqs = _inputs(body, shape, axis, sa, widths, 3)
    one = oracle.scan(body, init, seqs, axis=axis, state_axis=sa, reverse=reverse)
    many = oracle.scan_threads(body, init, seqs, axis=axis, state_axis=sa, reverse=reverse, threads=threads)
    assert many.dtype == np.float32 and many.shape == one.shape
    assert np.array_equal(many.view(np.uint32), one.view(np.uint32))
    g = np.random.default_rng(4).standard_normal(one.shape).astype(np.float32)
    gi1, gs1 = oracle.scan_backward(body, init, seqs, one, g, axis=axis, state_axis=sa, reverse=reverse)
    gim, gsm = oracle.scan_backward_threads(body, init, seqs, one, g, axis=axis, state_axis=sa, reverse=reverse,
                                            threads=threads)
    for p, q in zip([gi1] + gs1, [gim] + gsm):
        assert p.shape == q.shape and np.array_equal(p.view(np.uint32), q.view(np.uint32))


def test_lane_blocks_cover_dim0_once():
    for n in (1, 2, 7, 64, 262144):
        for k in (1, 3, 16, 100):
            blocks = oracle._lane_blocks(n, k)
            assert blocks[0][0] == 0 and blocks[-1][1] == n
            assert all(b[1] == c[0] for b, c in zip(blocks, blocks[1:]))
            assert len(blocks) == min(n, k) and all(hi > lo for lo, hi in blocks)
            sizes = [hi - lo for lo, hi in blocks]
            assert max(sizes) - min(sizes) <= 1


def test_threaded_oracle_rejects_what_the_oracle_rejects():
    init = np.zeros((4, 3), np.float32)
    x = np.zeros((4, 5, 3), np.float32)
    with pytest.raises(ValueError):
        oracle.scan_threads(oracle.TANH_DECAY, init[:, :2], [x, x], axis=1, threads=2)


def test_host_threads_is_positive():
    assert oracle.host_threads() >= 1


def test_split_rows_runs_each_block_once():
    for n, t in ((1, 4), (10, 3), (64, 16), (5, 64)):
        seen = []
        used = oracle.split_rows(lambda lo, hi: seen.append((lo, hi)), n, t)
        seen.sort()
        assert used == len(seen) == min(n, t)
        assert seen[0][0] == 0 and seen[-1][1] == n and all(a[1] == b[0] for a, b in zip(seen, seen[1:]))


def test_body_oracle_on_row_blocks_is_bit_identical():
    """The body-program oracle run over row blocks in threads (as the GPU
    tests run it at full size) gives the whole-array result bit for bit."""
    from oracle.body import scan_body
    text = "(lambda (h x a) (tanh (+ x (* a h))))"
    init, (x, a) = _inputs(oracle.TANH_DECAY, (9, 21, 6), 1, False, None, 8)
    whole = scan_body(text, init, [x, a], axis=1)
    out = np.empty_like(whole)

    def rows(lo, hi):
        out[lo:hi] = scan_body(text, init[lo:hi], [x[lo:hi], a[lo:hi]], axis=1)
    oracle.split_rows(rows, 9, 4)
    assert np.array_equal(out.view(np.uint32), whole.view(np.uint32))
