"""Host-side multi-process logic of bench.py on CPU: two gloo ranks agree on
the slowest rank's time (max) and on the whole-job element count (sum), and
the barrier works.  (Every GPU call on this pool uses one GPU; the N > 1
bench path differs from N = 1 only in this plumbing: each rank scans its own
batch, with no exchange of data.)"""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w, lr = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    mx = bench.max_over_ranks(dist, 10.0 + r)
    sm = bench.sum_over_ranks(dist, float(100 * (r + 1)))
    bench.barrier(dist)
    dist.destroy_process_group()
    q.put((r, w, lr, mx, sm))


def test_two_gloo_ranks_aggregate_like_the_bench():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1]
    for r, w, lr, mx, sm in out:
        assert w == 2 and lr == r
        assert mx == 11.0          # slowest rank
        assert sm == 300.0         # whole-job total


def test_single_process_needs_no_group():
    import bench
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert bench.sum_over_ranks(None, 2.0) == 2.0
