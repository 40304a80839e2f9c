#!/usr/bin/env python3
"""Benchmark of the element-scan library on one GB300 (or N, one process each).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole scan over one batch of the workload (every
direction the workload names).  Inputs are seeded synthetic tensors already
resident in HBM when the timed region starts; they are larger than the 129 MB
L2, so no flush is needed between steps.  Device time comes from CUDA events
on the launching stream; the timed region is bracketed by a barrier and a
synchronize on both sides and the slowest rank's time is used.  Rank 0 prints
one JSON line.

``e2e`` is the same metric end to end through the public API with host
buffers: every step copies its inputs from pinned host memory, scans, and
copies the states back.  ``cpu_baseline`` times the CPU oracle (test
infrastructure, a plain loop) on a bounded sample of the same workload.
``--impl reference`` times only that oracle, as the comparison arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "element-scan elements/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "elements/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
PATH_KERNEL = {"lane_tma": "k_lane_tma", "time_tma": "k_time_tma", "vec_tma": "k_vec_tma", "generic": "k_generic"}
PATH_KERNEL_BWD = {"lane_tma": "k_lane_bwd", "generic": "k_generic_bwd", "vec_tma": "k_vec_bwd",
                   "time_tma": "k_time_bwd"}
PATH_KERNEL_BODY_BWD = {"generic": "k_body_generic_bwd", "lane_tma": "k_body_lane_bwd", "vec_tma": "k_body_vec_bwd",
                        "time_tma": "k_body_time_bwd"}
# kernels compiled at run time from a body program
PATH_KERNEL_BODY = {"lane_tma": "k_body_lane", "time_tma": "k_body_time", "vec_tma": "k_body_vec",
                    "generic": "k_body_generic"}


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; timing only, no data exchange)

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    """The largest `value` over all ranks (the slowest rank's time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region

class NvmlReader:
    """Read-only NVML queries through ctypes (SM clock, its maximum, power
    draw, the active clock-event reasons) for the GPU a process runs on.
    Nothing here changes a setting of the GPU."""
    SM = 1                                  # NVML_CLOCK_SM
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40}

    def __init__(self, local_index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.handle = ctypes.c_void_p()
        bus = self._pci_bus_id(local_index)
        rc = 1
        if bus is not None:
            rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.handle))
        if rc != 0:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(self._physical_index(local_index), ctypes.byref(self.handle))
        if rc != 0:
            raise OSError("no NVML handle for the device")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")

    @staticmethod
    def _pci_bus_id(local_index):
        try:
            import torch
            p = torch.cuda.get_device_properties(local_index)
            return "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        except Exception:   # noqa: BLE001 -- older torch: fall back to the index
            return None

    @staticmethod
    def _physical_index(local_index):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_index < len(ids) and ids[local_index].isdigit():
            return int(ids[local_index])
        return local_index

    def sample(self):
        ct = self.ct
        sm, mx, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(self.handle, self.SM, ct.byref(sm))
        self.lib.nvmlDeviceGetMaxClockInfo(self.handle, self.SM, ct.byref(mx))
        self.lib.nvmlDeviceGetPowerUsage(self.handle, ct.byref(mw))
        self.reasons_fn(self.handle, ct.byref(rs))
        return float(sm.value), float(mx.value), mw.value / 1e3, int(rs.value)


class ClockSampler:
    """SM clock and throttle reasons sampled in a background thread while the
    bench runs: in-process NVML every `period_ms` (fast enough to land inside
    a timed region of a few milliseconds), else `nvidia-smi -lms`."""
    FIELDS = ("clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: float = 0.5):
        self.samples = []            # (time, sm MHz, max MHz, watts, set of reasons)
        self.proc = None
        self.thread = None
        self.source = None
        self._stop = threading.Event()
        try:
            self.nvml = NvmlReader(gpu_index)
            self.nvml.sample()
            self.source = "nvml every %.1f ms" % period_ms
            self.thread = threading.Thread(target=self._poll, args=(period_ms / 1e3,), daemon=True)
            self.thread.start()
            return
        except Exception:   # noqa: BLE001 -- no NVML here: nvidia-smi instead
            self.nvml = None
        cmd = ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + ",".join(self.FIELDS),
               "--format=csv,noheader,nounits", "-lms", "50"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.source = "nvidia-smi -lms 50"
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _poll(self, period):
        while not self._stop.is_set():
            try:
                sm, mx, w, bits = self.nvml.sample()
            except Exception:   # noqa: BLE001
                return
            names = {n for n, b in NvmlReader.REASON_BITS.items() if bits & b}
            self.samples.append((time.time(), sm, mx, w, names))
            time.sleep(period)

    def _read(self):
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                names = {n for n, v in zip(self.REASONS, parts[4:8]) if v.lower() == "active"}
                self.samples.append((time.time(), num(parts[0]), num(parts[1]), num(parts[2]), names))

    def stop(self):
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        if self.source is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "neither NVML nor nvidia-smi available"}
        inside = [p for p in self.samples if t0 <= p[0] <= t1]
        used, note = inside, "samples inside the timed region"
        if not inside:
            used = list(self.samples)
            note = "no sample inside the timed region; samples over warm-up and timed steps"
        sm = sorted(p[1] for p in used if p[1] is not None)
        mx = [p[2] for p in used if p[2] is not None]
        pw = [p[3] for p in used if p[3] is not None]
        reasons = set()
        for p in used:
            reasons |= p[4]
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "power_w_max": max(pw) if pw else None, "samples": len(used),
                "samples_in_timed_region": len(inside), "source": self.source, "note": note}


# ---------------------------------------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# the sources each kernel is built from (besides the shared device headers);
# a body-program kernel also depends on the compiler that writes its functor
# and on the host code that picks its launch configuration
_SHARED_SOURCES = ["es_ptx.cuh", "es_device.cuh", "es_internal.h"]
_BODY_SOURCES = ["skel_common.cuh", "es_body_compiler.cu", "es_body_api.cu", "es_jit.cu"]
KERNEL_SOURCES = {
    "k_lane_tma": ["k_lane_tma.cu"], "k_time_tma": ["k_time_tma.cu"], "k_vec_tma": ["k_vec_tma.cu"],
    "k_generic": ["k_generic.cu"], "k_generic_bwd": ["k_generic.cu"], "k_lane_bwd": ["k_lane_bwd.cu"],
    "k_vec_bwd": ["k_vec_bwd.cu"], "k_time_bwd": ["k_time_bwd.cu"],
    "k_body_lane": ["skel_lane.cuh"] + _BODY_SOURCES, "k_body_time": ["skel_time.cuh"] + _BODY_SOURCES,
    "k_body_vec": ["skel_vec.cuh"] + _BODY_SOURCES, "k_body_generic": ["skel_generic.cuh"] + _BODY_SOURCES,
    "k_body_generic_bwd": ["skel_generic_bwd.cuh"] + _BODY_SOURCES,
    "k_body_lane_bwd": ["skel_lane_bwd.cuh"] + _BODY_SOURCES,
    "k_body_vec_bwd": ["skel_vec_bwd.cuh", "skel_vec.cuh"] + _BODY_SOURCES,
    "k_body_time_bwd": ["skel_time_bwd.cuh"] + _BODY_SOURCES,
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the sources a kernel is built from: a profile taken before any
    of them changed no longer describes the kernel."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "element_scan_recurrences_gb300", "csrc")
    for name in KERNEL_SOURCES.get(kernel, sorted(os.listdir(csrc))) + _SHARED_SOURCES:
        h.update(name.encode())
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, or None when there is none or the kernel's sources changed since."""
    path = os.path.join(ROOT, "profiles", "%s_%s.md" % (kernel, workload))
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    s = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != kernel_source_hash(kernel):
        return None
    return int(m.group(1))


def plan_of(es, w, reverse):
    if w.text is not None:
        return es.Body(w.text).plan(w.shape, w.axis, w.shape[-1] if w.state_axis else 0,
                                    w.seq_widths if w.state_axis else None, reverse)
    return es.plan(w.body, w.shape, w.axis, w.shape[-1] if w.state_axis else 0,
                   w.seq_widths if w.state_axis else None, reverse)


def oracle_scan(w, init, seqs, reverse):
    """The CPU oracle on host arrays: the fixed-body oracle, or the body-program
    oracle for a workload given as text."""
    if w.text is not None:
        from oracle.body import scan_body
        return scan_body(w.text, init, seqs, axis=w.axis, state_axis=w.state_axis, reverse=reverse)
    import oracle
    return oracle.scan(w.body, init, seqs, axis=w.axis, state_axis=w.state_axis, reverse=reverse)


def oracle_backward(w, init, seqs, states, grad_out, reverse):
    """The CPU gradient oracle on host arrays (fixed body or body program)."""
    if w.text is not None:
        from oracle.body_grad import scan_body_backward
        return scan_body_backward(w.text, init, seqs, states, grad_out, axis=w.axis, state_axis=w.state_axis,
                                  reverse=reverse)
    import oracle
    return oracle.scan_backward(w.body, init, seqs, states, grad_out, axis=w.axis, state_axis=w.state_axis,
                                reverse=reverse)


def take_sample(w, init, seqs, target_elems: int, min_rows: int = 1):
    """Whole sequences of a leading block of lanes, about `target_elems` output
    values per direction: the first rows along dim 0, at least `min_rows` of
    them where dim 0 has that many (or, when one row is already larger and one
    row is asked for, the first positions of the last lane axis of row 0).
    Returns (initial, [sequences], elements, description)."""
    if w.ax == 0:
        raise ValueError("sampling needs a dimension before the sequence axis")
    per_row = w.elements // w.shape[0]
    if per_row <= target_elems or min_rows > 1:
        k = max(1, min_rows, min(w.shape[0], target_elems // per_row))
        k = min(k, w.shape[0])
        pick = lambda t: t[:k]
        desc = "first %d of %d rows along dim 0" % (k, w.shape[0])
        elems = k * per_row
    else:
        lane_dim = w.rank - 2 if w.state_axis else w.rank - 1
        n_last = w.shape[lane_dim]
        m = max(1, min(n_last, int(n_last * target_elems / per_row)))
        if w.state_axis:
            pick = lambda t: t[:1, ..., :m, :]
        else:
            pick = lambda t: t[:1, ..., :m]
        desc = "row 0 along dim 0, first %d of %d positions along dim %d" % (m, n_last, lane_dim)
        elems = per_row * m // n_last
    cpu = lambda t: pick(t).contiguous().cpu().numpy()
    return cpu(init), [cpu(t) for t in seqs], elems, desc


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def run_row_blocks(fn, n_rows: int, threads: int) -> int:
    """fn(lo, hi) over contiguous blocks of rows [0, n_rows), one thread a
    block (the oracles' foreign calls and numpy's array operations release the
    interpreter lock); returns the number of blocks."""
    k = max(1, min(threads, n_rows))
    bounds = [n_rows * i // k for i in range(k + 1)]
    blocks = [(bounds[i], bounds[i + 1]) for i in range(k) if bounds[i + 1] > bounds[i]]
    if len(blocks) == 1:
        fn(*blocks[0])
        return 1
    import concurrent.futures
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(blocks)) as pool:
        for f in [pool.submit(fn, lo, hi) for lo, hi in blocks]:
            f.result()
    return len(blocks)


def _timed(fn):
    t0 = time.perf_counter()
    r = fn()
    return time.perf_counter() - t0, r


def oracle_baseline(sample, step, budget_s: float, threads: int):
    """Both CPU figures of the oracle, each the median of 3 runs on a bounded
    sample of the workload: one thread, and every host core (lanes split into
    contiguous blocks, one per thread, each block the unchanged loop).
    ``sample(target_elems, min_rows)`` returns (ctx, elements, description);
    ``step(ctx, threads)`` runs the oracle once over the sample and returns
    the threads it used.  The two runs' sample sizes are chosen so that the
    whole measurement takes about `budget_s`."""
    per_run = max(0.05, budget_s / 7.0)
    ctx, e, _ = sample(1 << 18, 1)
    t, _ = _timed(lambda: step(ctx, 1))
    rate = e / max(t, 1e-6)
    ctx, e1, d1 = sample(max(1, int(rate * per_run)), 1)
    t1 = sorted(_timed(lambda: step(ctx, 1))[0] for _ in range(3))[1]
    r1 = e1 / t1
    ctx, en, dn = sample(max(1, int(r1 * threads * per_run)), threads)
    t, _ = _timed(lambda: step(ctx, threads))
    if t > 3 * per_run:
        # one block of lanes per thread is too much work: fewer, smaller rows
        ctx, en, dn = sample(max(1, int(en * per_run / t)), 1)
    runs = sorted(_timed(lambda: step(ctx, threads)) for _ in range(3))
    tn, used = runs[1]
    return {"value": en / tn, "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": "%s (%d elements), %d threads on contiguous blocks of lanes, median of 3" % (dn, en, used),
            "cpu_model": cpu_model(), "host_cores": threads, "median_of": 3,
            "one_thread": {"value": r1, "unit": UNIT, "cores": 1,
                           "sample": "%s (%d elements), one thread, median of 3" % (d1, e1)}}


def scan_sampler(w, init, seqs, backward: bool):
    """sample() and step() of `oracle_baseline` for an element-scan workload
    (fixed body or body program), forward or backward (the sample's forward
    states and an all-ones output gradient are made untimed)."""
    import numpy as np
    import oracle
    oracle.build()

    def sample(target, min_rows):
        ins, ss, elems, desc = take_sample(w, init, seqs, target, min_rows)
        prep = []
        if backward:
            for reverse in w.reverse:
                st = oracle_scan_threads(w, ins, ss, reverse, host_threads())
                prep.append((st, np.ones_like(st)))
        dirs = "+".join("reverse" if r else "forward" for r in w.reverse)
        return (ins, ss, prep), elems * len(w.reverse), "%s of the same workload, %s" % (desc, dirs)

    def step(ctx, threads):
        ins, ss, prep = ctx
        for k, reverse in enumerate(w.reverse):
            if backward:
                oracle_backward_threads(w, ins, ss, prep[k][0], prep[k][1], reverse, threads)
            else:
                oracle_scan_threads(w, ins, ss, reverse, threads)
        return max(1, min(threads, ins.shape[0] if ins.ndim else 1))
    return sample, step


def oracle_scan_threads(w, init, seqs, reverse, threads):
    """The oracle on `threads` contiguous blocks of lanes along dim 0."""
    if w.text is None:
        import oracle
        return oracle.scan_threads(w.body, init, seqs, axis=w.axis, state_axis=w.state_axis, reverse=reverse,
                                   threads=threads)
    import numpy as np
    from oracle.body import scan_body
    shape = list(seqs[0].shape)
    if w.state_axis:
        shape[-1] = init.shape[-1]
    out = np.empty(shape, np.float32)

    def blk(lo, hi):
        out[lo:hi] = scan_body(w.text, init[lo:hi], [s[lo:hi] for s in seqs], axis=w.axis,
                               state_axis=w.state_axis, reverse=reverse)
    run_row_blocks(blk, out.shape[0], threads)
    return out


def oracle_backward_threads(w, init, seqs, states, grad_out, reverse, threads):
    """The gradient oracle on `threads` contiguous blocks of lanes along dim 0."""
    if w.text is None:
        import oracle
        return oracle.scan_backward_threads(w.body, init, seqs, states, grad_out, axis=w.axis,
                                            state_axis=w.state_axis, reverse=reverse, threads=threads)
    from oracle.body_grad import scan_body_backward

    def blk(lo, hi):
        scan_body_backward(w.text, init[lo:hi], [s[lo:hi] for s in seqs], states[lo:hi], grad_out[lo:hi],
                           axis=w.axis, state_axis=w.state_axis, reverse=reverse)
    run_row_blocks(blk, states.shape[0], threads)


def cpu_oracle_rate(w, init, seqs, budget_s: float, backward: bool = False):
    """`cpu_baseline` of an element-scan workload: the oracle as it stands on
    bounded samples, one thread and all host cores."""
    sample, step = scan_sampler(w, init, seqs, backward)
    return oracle_baseline(sample, step, budget_s, host_threads())


def body_live_mask(w):
    """The sequences a body workload's backward reads (for its algorithmic
    bytes), from the library's generated VJP; None without the library."""
    if w.text is None:
        return None
    try:
        from element_scan_recurrences_gb300 import binding as es
        return es.Body(w.text).vjp_live_mask(w.shape[-1] if w.state_axis else 0,
                                             w.seq_widths if w.state_axis else None)
    except Exception:   # noqa: BLE001 -- metadata only
        return None


def reference_steps(args, sample, step, config):
    """--impl reference: the oracle on every host core as the comparison arm;
    each of the K timed steps (after W untimed ones) scans the same bounded
    sample of the workload, sized so that the whole run takes a few minutes."""
    threads = host_threads()
    step_budget = max(0.05, min(1.0, 120.0 / max(1, args.steps + args.warmup)))
    ctx, e, _ = sample(1 << 18, 1)
    t, _ = _timed(lambda: step(ctx, threads))
    rate = e / max(t, 1e-6)
    ctx, elems, desc = sample(max(1, int(rate * step_budget)), threads)
    t, _ = _timed(lambda: step(ctx, threads))
    if t > 3 * step_budget:
        ctx, elems, desc = sample(max(1, int(elems * step_budget / t)), 1)
    used = 1
    for _ in range(args.warmup):
        used = step(ctx, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(ctx, threads)
    dt = time.perf_counter() - t0
    value = elems * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": "%s (%d elements per step), %d threads on contiguous blocks of lanes" % (
                             desc, elems, used), "cpu_model": cpu_model(), "host_cores": threads},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args, w):
    """--impl reference for an element-scan workload (the fixed-body oracle,
    or the body-program oracle for a body given as text)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from element_scan_recurrences_gb300 import workloads as wl
    init, seqs = wl.make_inputs(w, "cpu")
    backward = args.pass_ == "backward"
    sample, step = scan_sampler(w, init, seqs, backward)
    return reference_steps(args, sample, step, config_of(w, backward, body_live_mask(w) if backward else None))


def config_of(w, backward=False, live=None):
    alg = w.backward_algorithmic_bytes(live) if backward else w.algorithmic_bytes()
    body = w.text if w.text is not None else ["TANH_DECAY", "NORMCAP", "MAXPLUS"][w.body]
    return {"workload": w.name + (" (backward pass)" if backward else ""),
            "pass": "backward" if backward else "forward", "body": body, "shape": list(w.shape),
            "axis": w.axis, "state_axis": w.state_axis, "seq_widths": list(w.seq_widths) if w.state_axis else None,
            "directions": ["reverse" if r else "forward" for r in w.reverse], "elements_per_step": w.elements *
            len(w.reverse), "algorithmic_bytes_per_step": alg * len(w.reverse),
            "l2": "no flush: inputs and outputs (%.2f GB) exceed the 129 MB L2" % (alg / 1e9)}


def time_device_steps(step, stream, device, dist, args, rank, local, es):
    """W untimed warm-up steps, then K timed steps bracketed by a barrier and a
    synchronize on both sides; CUDA events on the launching stream.  Returns
    (region ms over the slowest rank, per-step ms, kernel launches, clocks)."""
    import torch
    sampler = ClockSampler(local) if rank == 0 else None
    for _ in range(max(args.warmup, 0)):
        step()
    es.device_status(stream)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(dist, device)
    torch.cuda.synchronize(device)
    launches0 = es.launch_count()
    t_host0 = time.time()
    for i in range(args.steps):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(device)
    t_host1 = time.time()
    barrier(dist, device)
    launches = es.launch_count() - launches0
    es.device_status(stream)
    per_step_ms = [st.elapsed_time(e) for st, e in zip(starts, ends)]
    region_ms = max_over_ranks(dist, starts[0].elapsed_time(ends[-1]), device)
    clocks = None
    if sampler is not None:
        sampler.stop()
        clocks = sampler.summary(t_host0, t_host1)
    return region_ms, per_step_ms, launches, clocks


def chain_bound(es, w, program, stream, device, backward, sm_mhz):
    """The serial bound of a workload with few lanes: the same kernel on one
    CTA's worth of lanes (the first lanes of row 0, every trip), timed alone,
    where no other CTA competes for bandwidth.  Its time is T trips x the
    cycles one trip of the chain takes; the full launch cannot be faster than
    that however much bandwidth is left."""
    import torch
    from element_scan_recurrences_gb300 import workloads as wl
    W = w.shape[-1]
    per_warp = 32 * min(W, 4) // W if w.state_axis else 32
    lanes = 2 * per_warp                       # one CTA of two consumer warps
    shape = list(w.shape)
    shape[0] = 1
    shape[w.rank - 2 if w.state_axis else w.rank - 1] = lanes
    probe = w.with_shape(shape, name=w.name + "_one_cta")
    init, seqs = wl.make_inputs(probe, device)
    out = torch.empty(probe.shape, device=device)
    r = probe.reverse[0]
    if backward:
        if program is not None:
            program.scan_into(init, seqs, out, axis=w.axis, state_axis=w.state_axis, reverse=r, stream=stream)
        else:
            es.scan_into(w.body, init, seqs, out, axis=w.axis, state_axis=w.state_axis, reverse=r, stream=stream)
        g = torch.ones_like(out)
        grads = (torch.empty_like(init), [torch.empty_like(t) for t in seqs])

    def once():
        if backward:
            if program is not None:
                program.scan_backward(init, seqs, out, g, axis=w.axis, state_axis=w.state_axis, reverse=r,
                                      grads=grads, stream=stream)
            else:
                es.scan_backward(w.body, init, seqs, out, g, axis=w.axis, state_axis=w.state_axis, reverse=r,
                                 grads=grads, stream=stream)
        elif program is not None:
            program.scan_into(init, seqs, out, axis=w.axis, state_axis=w.state_axis, reverse=r, stream=stream)
        else:
            es.scan_into(w.body, init, seqs, out, axis=w.axis, state_axis=w.state_axis, reverse=r, stream=stream)

    for _ in range(3):
        once()
    times = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        once()
        e1.record(stream)
        torch.cuda.synchronize(device)
        times.append(e0.elapsed_time(e1))
    es.device_status(stream)
    ms = sorted(times)[len(times) // 2]
    res = {"latency_bound_ms": ms, "latency_probe": "the same kernel on %d lanes (one CTA), shape %s, median of 5"
           % (lanes, shape)}
    if sm_mhz:
        res["cycles_per_trip"] = ms * 1e-3 * sm_mhz * 1e6 / w.T
    return res


def time_e2e(e2e_step, steps, stream, device, dist):
    """One untimed end-to-end step, then `steps` timed ones (events on the
    stream the copies and kernels run on); ms over the slowest rank."""
    import torch
    e2e_step()
    torch.cuda.synchronize(device)
    barrier(dist, device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    barrier(dist, device)
    return max_over_ranks(dist, e0.elapsed_time(e1), device)


def roofline_of(kernel, prof_name, alg_bytes, kernel_ms):
    peak, peak_kind = measured_peaks()
    achieved = alg_bytes / (kernel_ms / 1e3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": profiled_traffic(kernel, prof_name), "kernel": kernel,
            "algorithmic_bytes_per_launch": alg_bytes, "kernel_ms": kernel_ms,
            "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs, copy burst)" % peak_kind
            if peak_kind == "measured" else "fallback 6.8 TB/s"}


def emit_line(args, world, value, region_ms, config, roofline, cpu, e2e, launches, clocks, path):
    """Rank 0's JSON line.  `config` is the same object the reference arm
    prints; the kernel path and the multi-GPU arrangement sit beside it."""
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": region_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config,
        "path": path, "parallelism": "replicas: each GPU scans its own batch" if world > 1 else "single GPU",
        "achieved_gbs": roofline["achieved"], "hbm_frac": roofline["frac"],
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def gpu_setup():
    import torch
    from element_scan_recurrences_gb300 import binding as es
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device; the library has no CPU path")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    es.lib()
    return es, rank, world, local, device, dist


def run_ours(args, w):
    import torch
    from element_scan_recurrences_gb300 import workloads as wl

    es, rank, world, local, device, dist = gpu_setup()
    # weak scaling: each rank scans its own batch of the workload (own seed)
    init, seqs = wl.make_inputs(w, device, seed=w.seed + rank)
    out = torch.empty(w.shape, device=device, dtype=torch.float32)
    outs = [out] + [torch.empty_like(out) for _ in w.reverse[1:]]
    stream = torch.cuda.current_stream(device)
    plans = [plan_of(es, w, r) for r in w.reverse]
    program = es.Body(w.text) if w.text is not None else None

    def scan_into(o, r):
        if program is not None:
            program.scan_into(init, seqs, o, axis=w.axis, state_axis=w.state_axis, reverse=r, stream=stream)
        else:
            es.scan_into(w.body, init, seqs, o, axis=w.axis, state_axis=w.state_axis, reverse=r, stream=stream)

    backward = args.pass_ == "backward"

    def scan_backward(o, g, gr, r):
        if program is not None:
            program.scan_backward(init, seqs, o, g, axis=w.axis, state_axis=w.state_axis, reverse=r, grads=gr,
                                  stream=stream)
        else:
            es.scan_backward(w.body, init, seqs, o, g, axis=w.axis, state_axis=w.state_axis, reverse=r, grads=gr,
                             stream=stream)

    if backward:
        # saved states and an output gradient per direction (untimed set-up)
        gen = torch.Generator(device=device)
        gen.manual_seed(1000 + rank)
        for o, r in zip(outs, w.reverse):
            scan_into(o, r)
        gouts = [torch.randn(w.shape, generator=gen, device=device) for _ in w.reverse]
        grads = [(torch.empty_like(init), [torch.empty_like(t) for t in seqs]) for _ in w.reverse]
        sw_, widths_ = (w.shape[-1], w.seq_widths) if w.state_axis else (0, None)
        if program is not None:
            plans = [program.plan_backward(w.shape, w.axis, sw_, widths_, r) for r in w.reverse]
        else:
            plans = [es.plan_backward(w.body, w.shape, w.axis, sw_, widths_, r) for r in w.reverse]

    def step():
        if backward:
            for o, g, gr, r in zip(outs, gouts, grads, w.reverse):
                scan_backward(o, g, gr, r)
            return
        for o, r in zip(outs, w.reverse):
            scan_into(o, r)

    region_ms, per_step_ms, launches, clocks = time_device_steps(step, stream, device, dist, args, rank, local, es)
    elems_step = w.elements * len(w.reverse)
    total_elems = sum_over_ranks(dist, float(elems_step * args.steps), device)
    value = total_elems / (region_ms / 1e3)
    kernel_ms = sum(per_step_ms) / len(per_step_ms) / len(w.reverse)

    # roofline of the dominant kernel (every launch of a step is the same kernel)
    live = None
    if backward and program is not None:
        live = program.vjp_live_mask(w.shape[-1] if w.state_axis else 0, w.seq_widths if w.state_axis else None)
    alg_bytes = w.backward_algorithmic_bytes(live) if backward else w.algorithmic_bytes()
    if backward:
        kernels = PATH_KERNEL_BODY_BWD if program is not None else PATH_KERNEL_BWD
    else:
        kernels = PATH_KERNEL_BODY if program is not None else PATH_KERNEL
    kernel = kernels.get(plans[0]["path"], plans[0]["path"])
    roofline = roofline_of(kernel, w.name + ("_backward" if backward else ""), alg_bytes, kernel_ms)
    if plans[0]["path"] == "vec_tma" and w.ax > 0 and rank == 0:
        roofline.update(chain_bound(es, w, program, stream, device, backward,
                                    clocks["sm_mhz"] if clocks and clocks.get("sm_mhz") else None))

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        init_h = init.cpu().pin_memory()
        seqs_h = [s.cpu().pin_memory() for s in seqs]
        out_h = [torch.empty(w.shape, dtype=torch.float32).pin_memory() for _ in w.reverse]
        h2d = (init_h.numel() + sum(s.numel() for s in seqs_h)) * 4
        d2h = sum(o.numel() for o in out_h) * 4
        e2e_steps = max(1, min(args.steps, args.e2e_steps))

        if backward:
            states_h = [o.cpu().pin_memory() for o in outs]
            gout_h = [g.cpu().pin_memory() for g in gouts]
            grads_h = [(torch.empty(init.shape).pin_memory(), [torch.empty(t.shape).pin_memory() for t in seqs])
                       for _ in w.reverse]
            h2d = (init_h.numel() + sum(t.numel() for t in seqs_h) + 2 * w.elements) * 4
            d2h = (init_h.numel() + sum(t.numel() for t in seqs_h)) * 4

        def e2e_step():
            if backward:
                # inputs, saved states and output gradient in; the three gradients out
                with torch.cuda.stream(stream):
                    for sh, gh, od, gd, gr_h, gr_d, r in zip(states_h, gout_h, outs, gouts, grads_h, grads,
                                                              w.reverse):
                        init.copy_(init_h, non_blocking=True)
                        for d, hh in zip(seqs, seqs_h):
                            d.copy_(hh, non_blocking=True)
                        od.copy_(sh, non_blocking=True)
                        gd.copy_(gh, non_blocking=True)
                        scan_backward(od, gd, gr_d, r)
                        gr_h[0].copy_(gr_d[0], non_blocking=True)
                        for hh, d in zip(gr_h[1], gr_d[1]):
                            hh.copy_(d, non_blocking=True)
                return
            for oh, od, r in zip(out_h, outs, w.reverse):
                if program is not None:
                    program.scan_host(init_h, seqs_h, oh, (init, seqs, od), axis=w.axis, state_axis=w.state_axis,
                                      reverse=r, stream=stream)
                else:
                    es.scan_host(w.body, init_h, seqs_h, oh, (init, seqs, od), axis=w.axis,
                                 state_axis=w.state_axis, reverse=r, stream=stream)

        e_ms = time_e2e(e2e_step, e2e_steps, stream, device, dist)
        e2e = {"value": sum_over_ranks(dist, float(elems_step * e2e_steps), device) / (e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": h2d * (len(w.reverse)), "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "ms_per_step": e_ms / e2e_steps}
        del init_h, seqs_h, out_h

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_rate(w, init, seqs, args.cpu_budget, backward=backward)

    if rank == 0:
        emit_line(args, world, value, region_ms, config_of(w, backward, live), roofline, cpu, e2e, launches,
                  clocks, plans[0]["path"])
    if dist is not None:
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# matrix-scan / linear-scan workloads

MATRIX_KERNEL = {"mat_tma": "k_mat_tma", "generic": "k_mat_generic", "lane_tma": "k_body_lane",
                 "time_tma": "k_body_time", "mat_chunked": "k_mat_chunk_final",
                 "mat_chunked_tma": "k_mat_tma_chunked"}
KERNEL_SOURCES.update({k: ["k_matrix.cu", "es_matrix_api.cu"]
                       for k in ("k_mat_tma", "k_mat_generic", "k_mat_chunk_final", "k_mat_tma_chunked")})


def matrix_scan_call(es, w, a, b, out, reverse, stream, workspace=None):
    if w.kind == "linear":
        es.linear_scan(a, b, axis=w.axis, reverse=reverse, out=out, stream=stream)
    elif workspace is not None:
        es.matrix_scan_ws(a, b, workspace, axis=w.axis, reverse=reverse, projective=w.projective, out=out,
                          stream=stream)
    else:
        es.matrix_scan(a, b, axis=w.axis, reverse=reverse, projective=w.projective, out=out, stream=stream)


def matrix_plan(es, w, reverse):
    if w.kind == "linear":
        return es.plan_linear_scan(w.a_shape, w.b_shape, w.axis, reverse)
    return es.plan_matrix_scan(w.a_shape, w.b_shape, w.axis, reverse, w.projective)


TABLE_KERNEL = {"time_tma": "k_table_time", "lane_tma": "k_table_lane", "generic": "k_table_generic"}
KERNEL_SOURCES.update({k: ["k_table.cu", "es_table_api.cu"] for k in TABLE_KERNEL.values()})


def table_config(w):
    alg = w.algorithmic_bytes()
    return {"workload": w.name, "pass": "forward", "op": "table-scan", "shape": list(w.shape), "axis": w.axis,
            "states": w.n_states, "symbols": w.n_syms, "dtype": "i32",
            "elements_per_step": w.elements, "algorithmic_bytes_per_step": alg,
            "l2": "no flush: symbols and states (%.2f GB) exceed the 129 MB L2" % (alg / 1e9)}


def matrix_config(w, backward=False):
    alg = w.backward_algorithmic_bytes() if backward else w.algorithmic_bytes()
    return {"workload": w.name + (" (backward pass)" if backward else ""),
            "pass": "backward" if backward else "forward", "op": "linear-scan" if w.kind == "linear" else "matrix-scan",
            "a_shape": list(w.a_shape), "b_shape": list(w.b_shape), "axis": w.axis, "n": w.n, "m": w.m,
            "projective": w.projective, "workspace": getattr(w, "workspace", False),
            "directions": ["reverse" if r else "forward" for r in w.reverse],
            "elements_per_step": w.elements * len(w.reverse), "algorithmic_bytes_per_step": alg * len(w.reverse),
            "l2": "no flush: inputs and outputs (%.2f GB) exceed the 129 MB L2" % (alg / 1e9)}


def matrix_sample(w, a, b, target_elems, min_rows=1):
    """The first rows along dim 0 (every lane of them, whole sequences) of a
    and b, about `target_elems` output values and at least `min_rows` rows
    where dim 0 has them; when that is already larger and the scan runs along
    dim 1 (few long lanes), the first trips of those rows."""
    per_row = w.elements // w.lead[0]
    rows = max(1, min(w.lead[0], min_rows))
    if w.ax != 1 or per_row * rows <= target_elems:
        k = max(rows, min(w.lead[0], target_elems // per_row))
        return (a[:k].contiguous().cpu().numpy(), b[:k].contiguous().cpu().numpy(), k * per_row,
                "first %d of %d rows along dim 0" % (k, w.lead[0]))
    per_trip = per_row // w.T
    t = max(1, min(w.T, target_elems // (per_trip * rows)))
    return (a[:rows, :t].contiguous().cpu().numpy(), b[:rows, :t].contiguous().cpu().numpy(), rows * t * per_trip,
            "first %d of %d rows along dim 0, their first %d of %d trips" % (rows, w.lead[0], t, w.T))


def matrix_oracle(w, a, b, reverse):
    import oracle.matrix as M
    if w.kind == "linear":
        return M.linear_scan(a, b, axis=w.axis, reverse=reverse)
    return M.matrix_scan(a, b, axis=w.axis, reverse=reverse, projective=w.projective)


def matrix_oracle_backward(w, a, b, states, grad_out, reverse):
    import oracle.matrix as M
    if w.kind == "linear":
        return M.linear_scan_backward(a, b, states, grad_out, axis=w.axis, reverse=reverse)
    return M.matrix_scan_backward(a, b, states, grad_out, axis=w.axis, reverse=reverse)


def matrix_backward_call(es, w, a, b, states, grad_out, grads, reverse, stream, workspace=None):
    if w.kind == "linear":
        es.linear_scan_backward(a, b, states, grad_out, axis=w.axis, reverse=reverse, grads=grads, stream=stream)
    elif workspace is not None:
        es.matrix_scan_backward_ws(a, b, states, grad_out, workspace, axis=w.axis, reverse=reverse, grads=grads,
                                   stream=stream)
    else:
        es.matrix_scan_backward(a, b, states, grad_out, axis=w.axis, reverse=reverse, grads=grads, stream=stream)


def matrix_backward_plan(es, w, reverse, workspace=None):
    if w.kind == "linear":
        return es.plan_linear_scan_backward(w.a_shape, w.b_shape, w.axis, reverse)
    if workspace is not None:
        return es.plan_matrix_scan_backward_ws(w.a_shape, w.b_shape, workspace.numel(), w.axis, reverse)
    return es.plan_matrix_scan_backward(w.a_shape, w.b_shape, w.axis, reverse)


# the backward's dominant kernels: linear-scan runs the element-scan backward
# skeletons of its body; matrix-scan two launches (the cotangent scan on a's
# transposes, then grad_a), timed as one call
MATRIX_BWD_KERNEL = {"mat_tma": "k_mat_tma_bwd", "generic": "k_mat_generic_bwd",
                     "lane_tma": "k_body_lane_bwd", "time_tma": "k_body_time_bwd",
                     "mat_chunked_tma": "k_mat_tma_chunked_bwd"}
KERNEL_SOURCES.update({k: ["k_matrix.cu", "es_matrix_api.cu"]
                       for k in ("k_mat_tma_bwd", "k_mat_generic_bwd", "k_mat_tma_chunked_bwd")})


def op_sample(w, inputs, target_elems, min_rows=1):
    """A bounded sample of an op workload for the oracle: (inputs, elements,
    description)."""
    from element_scan_recurrences_gb300 import workloads as wl
    if isinstance(w, wl.TableWorkload):
        table, sym = inputs
        per_row = w.elements // w.shape[0]
        k = min(w.shape[0], max(1, min_rows, target_elems // per_row))
        return ([table.cpu().numpy(), sym[:k].contiguous().cpu().numpy()], k * per_row,
                "first %d of %d rows along dim 0" % (k, w.shape[0]))
    sa, sb, elems, desc = matrix_sample(w, inputs[0], inputs[1], target_elems, min_rows)
    return [sa, sb], elems, desc


def op_oracle(w, inputs, reverse):
    from element_scan_recurrences_gb300 import workloads as wl
    if isinstance(w, wl.TableWorkload):
        import oracle.table as TS
        return TS.table_scan(inputs[0], inputs[1], axis=w.axis)
    return matrix_oracle(w, inputs[0], inputs[1], reverse)


def op_backward_prep(w, sample):
    """The sample's saved states and an all-ones state gradient per
    direction (made before any timing)."""
    import numpy as np
    prep = []
    for r in w.reverse:
        st = op_oracle(w, sample, r)
        prep.append((st, np.ones_like(st)))
    return prep


def op_sampler(w, inputs, backward):
    """sample() and step() of `oracle_baseline` for a matrix-scan,
    linear-scan or table-scan workload; the threads split the sample's rows
    along dim 0 into contiguous blocks (one thread when the scan runs along
    dim 0)."""
    from element_scan_recurrences_gb300 import workloads as wl
    table = isinstance(w, wl.TableWorkload)

    def sample(target, min_rows):
        smp, elems, desc = op_sample(w, inputs, target, min_rows)
        prep = op_backward_prep(w, smp) if backward else None
        return (smp, prep), elems * len(w.reverse), "%s of the same workload" % desc

    def step(ctx, threads):
        smp, prep = ctx
        rows = smp[1].shape[0]
        if w.ax == 0 or rows <= 1:
            threads = 1
        used = 1
        for k, r in enumerate(w.reverse):
            if table:
                fn = lambda lo, hi: op_oracle(w, [smp[0], smp[1][lo:hi]], r)
            elif backward:
                fn = lambda lo, hi: matrix_oracle_backward(w, smp[0][lo:hi], smp[1][lo:hi], prep[k][0][lo:hi],
                                                           prep[k][1][lo:hi], r)
            else:
                fn = lambda lo, hi: matrix_oracle(w, smp[0][lo:hi], smp[1][lo:hi], r)
            if threads > 1:
                used = run_row_blocks(fn, rows, threads)
            else:
                fn(0, rows)
        return used
    return sample, step


def op_cpu_rate(w, inputs, budget_s, backward=False):
    """`cpu_baseline` of an op workload: its oracle on bounded samples, one
    thread and all host cores."""
    sample, step = op_sampler(w, inputs, backward)
    return oracle_baseline(sample, step, budget_s, host_threads())


class OpJob:
    """What the bench needs of a matrix-scan, linear-scan or table-scan
    workload: its device inputs, one launch per direction, the plan, the
    oracle on a sample, the configuration."""

    def __init__(self, es, w, device, seed):
        from element_scan_recurrences_gb300 import workloads as wl
        self.es, self.w = es, w
        self.table = isinstance(w, wl.TableWorkload)
        if self.table:
            self.inputs = list(wl.make_table_inputs(w, device, seed=seed))
            self.out_shape, self.out_dtype = w.shape, "int32"
            self.kernels = TABLE_KERNEL
        else:
            import torch
            self.inputs = list(wl.make_matrix_inputs(w, device, seed=seed))
            self.out_shape, self.out_dtype = w.b_shape, "float32"
            self.kernels = MATRIX_KERNEL
            self.workspace = None
            if getattr(w, "workspace", False):
                nbytes = es.matrix_scan_workspace(w.a_shape, w.b_shape, w.axis, w.projective)
                self.workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)

    def call(self, inputs, out, reverse, stream):
        es, w = self.es, self.w
        if self.table:
            es.table_scan(inputs[0], inputs[1], axis=w.axis, out=out, stream=stream)
        else:
            matrix_scan_call(es, w, inputs[0], inputs[1], out, reverse, stream, self.workspace)

    def plan(self, reverse):
        es, w = self.es, self.w
        if self.table:
            return es.plan_table_scan(w.n_states, w.n_syms, w.shape, w.axis)
        if self.workspace is not None:
            return es.plan_matrix_scan_ws(w.a_shape, w.b_shape, self.workspace.numel(), w.axis, reverse,
                                          w.projective)
        return matrix_plan(es, w, reverse)

    def launches_per_call(self):
        return 3 if self.plan(False)["path"] in ("mat_chunked", "mat_chunked_tma") else 1

    def config(self):
        return table_config(self.w) if self.table else matrix_config(self.w)


def run_ours_op(args, w):
    import torch

    es, rank, world, local, device, dist = gpu_setup()
    job = OpJob(es, w, device, w.seed + rank)
    dtype = getattr(torch, job.out_dtype)
    outs = [torch.empty(job.out_shape, device=device, dtype=dtype) for _ in w.reverse]
    stream = torch.cuda.current_stream(device)
    plans = [job.plan(r) for r in w.reverse]
    backward = args.pass_ == "backward"
    if backward:
        # saved states and a state gradient per direction (untimed set-up)
        for o, r in zip(outs, w.reverse):
            job.call(job.inputs, o, r, stream)
        gen = torch.Generator(device=device)
        gen.manual_seed(1000 + rank)
        gouts = [torch.randn(job.out_shape, generator=gen, device=device) for _ in w.reverse]
        grads = [(torch.empty_like(job.inputs[0]), torch.empty_like(job.inputs[1])) for _ in w.reverse]
        plans = [matrix_backward_plan(es, w, r, job.workspace) for r in w.reverse]

    def step():
        if backward:
            for o, g, gr, r in zip(outs, gouts, grads, w.reverse):
                matrix_backward_call(es, w, job.inputs[0], job.inputs[1], o, g, gr, r, stream, job.workspace)
            return
        for o, r in zip(outs, w.reverse):
            job.call(job.inputs, o, r, stream)

    region_ms, per_step_ms, launches, clocks = time_device_steps(step, stream, device, dist, args, rank, local, es)
    elems_step = w.elements * len(w.reverse)
    value = sum_over_ranks(dist, float(elems_step * args.steps), device) / (region_ms / 1e3)
    kernel_ms = sum(per_step_ms) / len(per_step_ms) / len(w.reverse)
    if backward:
        kernel = MATRIX_BWD_KERNEL.get(plans[0]["path"], plans[0]["path"])
        roofline = roofline_of(kernel, w.name + "_backward", w.backward_algorithmic_bytes(), kernel_ms)
        if w.kind != "linear" and plans[0]["path"] == "mat_chunked_tma":
            roofline["kernel"] = ("k_mat_tma (transposed, chunk pass) + k_mat_chunk_link + k_mat_tma (transposed, "
                                  "final pass) + k_mat_da")
            roofline["note"] = ("a call of four launches timed as one: the cotangent scan chunked (a and grad_out read "
                                "by both scan passes), then grad_a from the cotangent and the saved states")
        elif w.kind != "linear":
            roofline["kernel"] = "k_mat_%s (transposed) + k_mat_da" % ("tma" if plans[0]["path"] == "mat_tma"
                                                                      else "generic")
            roofline["note"] = ("a call timed as one: the cotangent scan on a's transposes and grad_a from the "
                                "cotangent and the saved states (on the TMA path in windows of trips, each window's "
                                "grad_a beside the next scan window on a second stream); the cotangent is written "
                                "and read again, so its DRAM traffic is up to (2n^2 + 4nm) / (2n^2 + 3nm) of the "
                                "algorithmic bytes, less where a window's cotangent is read back from L2")
    else:
        kernel = job.kernels.get(plans[0]["path"], plans[0]["path"])
        roofline = roofline_of(kernel, w.name, w.algorithmic_bytes(), kernel_ms)
    if not backward and plans[0]["path"] in ("mat_chunked", "mat_chunked_tma"):
        # three launches make one call: `achieved` is the whole call's
        # algorithmic bytes over its time
        roofline["kernel"] = ("k_mat_tma (chunk pass) + k_mat_chunk_link + k_mat_tma (final pass)"
                              if plans[0]["path"] == "mat_chunked_tma" else
                              "k_mat_chunk_local + k_mat_chunk_carry + k_mat_chunk_final")
        roofline["kernel_ms"] = kernel_ms
        roofline["note"] = ("a call of three launches timed as one; its DRAM traffic is about 5/3 of the "
                            "algorithmic bytes (a and b are read in the first and the last pass)")

    e2e = None
    if not args.no_e2e:
        hosts = [t.cpu().pin_memory() for t in job.inputs]
        out_h = [torch.empty(job.out_shape, dtype=dtype).pin_memory() for _ in w.reverse]
        e2e_steps = max(1, min(args.steps, args.e2e_steps))

        h2d = sum(t.numel() for t in hosts) * 4 * len(w.reverse)
        d2h = sum(o.numel() for o in out_h) * 4
        if backward:
            states_h = [o.cpu().pin_memory() for o in outs]
            gout_h = [g.cpu().pin_memory() for g in gouts]
            grads_h = [(torch.empty(job.inputs[0].shape).pin_memory(), torch.empty(job.inputs[1].shape).pin_memory())
                       for _ in w.reverse]
            h2d = (sum(t.numel() for t in hosts) + 2 * w.elements) * 4 * len(w.reverse)
            d2h = (job.inputs[0].numel() + job.inputs[1].numel()) * 4 * len(w.reverse)

        def e2e_step():
            with torch.cuda.stream(stream):
                if backward:
                    # inputs, saved states and state gradient in; both gradients out
                    for sh, gh, od, gd, gr_h, gr_d, r in zip(states_h, gout_h, outs, gouts, grads_h, grads,
                                                              w.reverse):
                        for d, hh in zip(job.inputs, hosts):
                            d.copy_(hh, non_blocking=True)
                        od.copy_(sh, non_blocking=True)
                        gd.copy_(gh, non_blocking=True)
                        matrix_backward_call(es, w, job.inputs[0], job.inputs[1], od, gd, gr_d, r, stream,
                                             job.workspace)
                        gr_h[0].copy_(gr_d[0], non_blocking=True)
                        gr_h[1].copy_(gr_d[1], non_blocking=True)
                    return
                for oh, od, r in zip(out_h, outs, w.reverse):
                    for d, hh in zip(job.inputs, hosts):
                        d.copy_(hh, non_blocking=True)
                    job.call(job.inputs, od, r, stream)
                    oh.copy_(od, non_blocking=True)

        e_ms = time_e2e(e2e_step, e2e_steps, stream, device, dist)
        e2e = {"value": sum_over_ranks(dist, float(elems_step * e2e_steps), device) / (e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "ms_per_step": e_ms / e2e_steps}
        del hosts, out_h

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = op_cpu_rate(w, job.inputs, args.cpu_budget, backward=backward)
    if rank == 0:
        emit_line(args, world, value, region_ms, matrix_config(w, True) if backward else job.config(), roofline,
                  cpu, e2e, launches, clocks, plans[0]["path"])
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_reference_op(args, w):
    """--impl reference for a matrix-scan, linear-scan or table-scan
    workload: its oracle on every host core over a bounded sample of the same
    workload, each step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from element_scan_recurrences_gb300 import workloads as wl
    if isinstance(w, wl.TableWorkload):
        inputs = list(wl.make_table_inputs(w, "cpu"))
        config = table_config(w)
    else:
        inputs = list(wl.make_matrix_inputs(w, "cpu"))
        config = matrix_config(w)
    backward = args.pass_ == "backward"
    if backward:
        config = matrix_config(w, True)
    sample, step = op_sampler(w, inputs, backward)
    return reference_steps(args, sample, step, config)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="tanh_decay_lanes")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--pass", dest="pass_", choices=["forward", "backward"], default="forward",
                    help="time the scan or its backward pass (gradients from saved states)")
    ap.add_argument("--cpu-budget", type=float, default=8.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--trips", type=int, default=0,
                    help="profiling aid: shorten the sequence axis to this many trips (same lanes, same kernel "
                         "launch shape); lines printed with it are not the workload's bench numbers")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    from element_scan_recurrences_gb300 import workloads as wl
    ops = dict(wl.MATRIX_WORKLOADS, **wl.TABLE_WORKLOADS)
    if args.workload in ops:
        w = ops[args.workload]
        if args.trips:
            w = w.with_trips(args.trips)
        if args.pass_ == "backward" and w.name in wl.TABLE_WORKLOADS:
            ap.error("--pass backward: table-scan states have no gradient")
        return run_reference_op(args, w) if args.impl == "reference" else run_ours_op(args, w)
    w = wl.WORKLOADS[args.workload]
    if args.trips:
        shape = list(w.shape)
        shape[w.ax] = args.trips
        w = w.with_shape(shape, name="%s_T%d" % (w.name, args.trips))
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
