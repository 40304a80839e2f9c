"""Host-side pieces of bench.py on CPU: the oracle's two baseline figures
(one thread and all host cores, median of 3, with the CPU model), the row
sampling, the thread blocks, and that both arms print the same `config`."""
import json

import bench
from element_scan_recurrences_gb300 import workloads as wl


def test_row_blocks_cover_every_row_once():
    for n in (1, 5, 64):
        for t in (1, 3, 8, 100):
            seen = []
            used = bench.run_row_blocks(lambda lo, hi: seen.append((lo, hi)), n, t)
            seen.sort()
            assert used == len(seen) == min(n, t)
            assert seen[0][0] == 0 and seen[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(seen, seen[1:]))


def test_take_sample_honours_min_rows():
    w = wl.custom(wl.TANH_DECAY, (12, 16, 8), 1)
    init, seqs = wl.make_inputs(w, "cpu")
    ins, ss, elems, desc = bench.take_sample(w, init, seqs, 1, min_rows=5)
    assert ins.shape == (5, 8) and ss[0].shape == (5, 16, 8) and elems == 5 * 16 * 8
    ins, ss, elems, _ = bench.take_sample(w, init, seqs, 10 ** 9, min_rows=5)
    assert ss[0].shape == (12, 16, 8)


def test_cpu_baseline_has_both_figures():
    w = wl.custom(wl.TANH_DECAY, (16, 64, 32), 1)
    init, seqs = wl.make_inputs(w, "cpu")
    cpu = bench.cpu_oracle_rate(w, init, seqs, budget_s=0.3)
    assert cpu["kind"] == "oracle" and cpu["median_of"] == 3 and cpu["value"] > 0
    assert cpu["one_thread"]["cores"] == 1 and cpu["one_thread"]["value"] > 0
    assert 1 <= cpu["cores"] <= cpu["host_cores"] == bench.host_threads()
    if bench.host_threads() > 1:
        assert cpu["cores"] > 1
    assert isinstance(cpu["cpu_model"], str) and cpu["cpu_model"]


def test_op_baseline_runs_on_row_blocks():
    w = wl.MATRIX_WORKLOADS["matrix_scan_delta_rule"].with_trips(8)
    a, b = wl.make_matrix_inputs(w, "cpu")
    cpu = bench.op_cpu_rate(w, [a, b], budget_s=0.3)
    assert cpu["value"] > 0 and cpu["one_thread"]["value"] > 0 and cpu["cores"] >= 1


def test_reference_arm_prints_the_same_config(capsys):
    w = wl.WORKLOADS["tanh_decay_small"]
    args = bench.main.__globals__["argparse"].Namespace(steps=3, warmup=3, gpus=1, pass_="forward")
    assert bench.run_reference(args, w.with_shape((16, 64, 8), name=w.name)) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["cpu_baseline"]["cores"] >= 1
    assert line["config"] == bench.config_of(w.with_shape((16, 64, 8), name=w.name))
    assert "path" not in line["config"] and "parallelism" not in line["config"]
