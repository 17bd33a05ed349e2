#!/usr/bin/env python3
"""Benchmark of row-wise ArgMax/ArgMin on one GB300 (or N replicas).

Workload (the default line): the wide-row sampler-logit group, i.e. ArgMax and
ArgMin over [1, 202048] and [1, 262144] rows, fp32 and bf16, each with a unique
planted extreme and with a duplicated one: 16 calls. One *step* is those 16
calls, each on its own input already resident in HBM. Inputs are rotated over
enough copies that the bytes touched between two reuses of a copy exceed the
L2 cache, so every call reads from HBM. The steps are replayed as CUDA graphs
(one per input copy) so that the device time is not host-bound.

Metric: microseconds per call (lower is better) and achieved HBM GB/s of the
algorithmic bytes (rows*cols*elem read + rows*8 written), against the measured
copy bandwidth of this GPU.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--no-configs] [--no-cpu-baseline] [--workload NAME]

One JSON line on stdout (rank 0).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

L2_BYTES = 129 * 2**20
FALLBACK_HBM_GBS = 6800.0
METRIC = "ArgMax/ArgMin µs/call and achieved HBM GB/s (% of GB300 peak) per [rows,cols]"
WORKLOADS = {
    # name -> (workload group, description)
    "wide_rows": (2, "ArgMax+ArgMin fp32+bf16 [1,202048]+[1,262144], unique and duplicated planted extreme"),
    "logits_32000": (1, "ArgMax fp32 [1,32000]"),
    "batches": (3, "ArgMax fp16/bf16/fp32 [8,202048]+[32,202048]"),
    "uniform_special": (4, "ArgMin/ArgMax fp32/f64 [4096,4096]+[65536,1024] with special rows"),
    "narrow": (5, "ArgMax fp32 [65536,64]+[4096,8]+[4096,128]"),
    "wide_rows_last": (-2, "the wide_rows cases with ties to the last index (ONNX select_last_index = 1)"),
    "axis": (6, "ArgMax/ArgMin over a non-last axis: [1,100000,1000], [1,1000,100000], [64,512,256] bf16, "
                "[128,4096,8], [16,2048,384] f64"),
    "cum": (7, "cummax/cummin with indices: [1,65536], [1,262144], [64,1024], [1024,64] int64, [4,16384] int32, "
               "[1,65536] f32/f64, [256,256] bf16"),
    "cum_large": (8, "cummax/cummin with indices at bandwidth scale: [1,2^24] int64, [16,2^20] f64, [4096,4096] f32, "
                     "[256,65536] f32"),
}
DTYPE_LABEL = {"f32": "f32", "f16": "f16", "bf16": "bf16", "f64": "f64", "i32": "i32", "i64": "i64"}
KERNEL_OF_PATH = {"rows": "rows_kernel", "split": "split_kernel", "cluster": "cluster_push_kernel", "axis": "axis_kernel",
                  "stream": "stream_kernel", "cum": "cum_kernel", "cum_split": "cum_split_kernel", "none": "none"}


def workload_cases(group: int):
    """Cases of a workload group; a negative group is the last-index variant."""
    if group > 0:
        return W.config_cases(group)
    return [dataclasses.replace(c, op=c.op + "_last", name=c.name + "_last") for c in W.config_cases(-group)]


def is_scan(c: W.Case) -> bool:
    return c.recipe == "cum_values"


def algo_bytes(c: W.Case, with_values: bool = False) -> int:
    """Algorithmic bytes of one call: the input read once, int64 indices
    written (one per row, per (outer, inner) column, or per element for the
    cummax/cummin scan, which also writes one value per element)."""
    es = W.ELEM_SIZE[c.dtype]
    if is_scan(c):
        return c.rows * c.cols * (2 * es + 8)
    outputs = c.rows * c.inner
    return c.rows * c.cols * c.inner * es + outputs * 8 + (outputs * es if with_values else 0)


def n_outputs(c: W.Case) -> int:
    return c.rows * c.cols if is_scan(c) else c.rows * c.inner


class CubCalls:
    """cub::DeviceReduce::ArgMax/ArgMin on single-row cases (timing
    comparison): one temporary buffer and one extremum slot per case."""

    def __init__(self, torch, cases):
        from row_wise_arg_gb300 import cub_compare
        self.C = cub_compare
        assert all(c.rows == 1 and c.inner == 1 and c.op in ("max", "min") and not is_scan(c) for c in cases)
        self.temp = [torch.empty(max(self.C.temp_bytes(c.dtype, c.op, c.cols), 16), dtype=torch.uint8, device="cuda")
                     for c in cases]
        self.val = [torch.empty(16, dtype=torch.uint8, device="cuda") for _ in cases]

    def __call__(self, i, c, x, out_idx, stream):
        self.C.argreduce_raw(x.data_ptr(), c.dtype, c.op, c.cols, self.val[i].data_ptr(), out_idx.data_ptr(),
                             self.temp[i].data_ptr(), self.temp[i].numel(), stream.cuda_stream)


class ThreadPerRowCalls:
    """The thread-per-row kernel (one thread scans a whole row: the pages'
    narrow-row design) as a forced plan of the same library, for the narrow
    configs' comparison: scalar loads as on the pages, or 16-byte vector
    loads (`vec`, rows 16-byte aligned), 256 threads, 4 loads in flight."""

    def __init__(self, A, cases, vec):
        from row_wise_arg_gb300 import _lib
        self.A = A
        self.plans = []
        for c in cases:
            p = _lib.argr_plan()
            p.path, p.block, p.group, p.vec, p.unroll = _lib.ARGR_PATH_ROWS, 256, 1, int(vec), 4
            p.flags = _lib.ARGR_PLAN_PDL
            p.blocks_per_row = 1
            p.grid_rows = min(-(-c.rows // 256), 65535)
            self.plans.append(p)

    def __call__(self, i, c, x, out_idx, stream):
        self.A.argreduce_with_plan(self.plans[i], x.view(c.rows, c.cols), c.op, dtype=c.dtype, out_idx=out_idx,
                                   stream=stream)


def cub_comparable(cases) -> bool:
    return all(c.rows == 1 and c.inner == 1 and c.op in ("max", "min") and not is_scan(c) for c in cases)


def call(A, c: W.Case, x, out_idx, scratch, stream, out_val=None):
    """One library call for case c on device data x (flat)."""
    if is_scan(c):
        A.argreduce_cum(x.view(c.rows, c.cols), c.op, dtype=c.dtype, out_idx=out_idx, out_val=out_val,
                        stream=stream)
    elif c.inner > 1:
        A.argreduce_axis(x.view(c.rows, c.cols, c.inner), 1, c.op, dtype=c.dtype, out_idx=out_idx, scratch=scratch,
                         stream=stream)
    else:
        A.argreduce(x.view(c.rows, c.cols), c.op, dtype=c.dtype, out_idx=out_idx, scratch=scratch, stream=stream)


def load_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# The sources each workload's kernels and launch plans are built from; a
# committed traffic figure is used only while they are unchanged.
_COMMON_SOURCES = ("device_common.cuh", "kernels_impl.cuh", "tma.cuh", "internal.h")
_WORKLOAD_SOURCES = {
    "argreduce": _COMMON_SOURCES + ("plan.cpp", "kernels_f32.cu", "kernels_f16.cu", "kernels_bf16.cu",
                                    "kernels_f64.cu"),
    "axis": _COMMON_SOURCES + ("plan.cpp", "axis_f32.cu", "axis_f16.cu", "axis_bf16.cu", "axis_f64.cu"),
    "cum": _COMMON_SOURCES + ("plan_cum.cpp", "cum_impl.cuh", "cum_f32.cu", "cum_f16.cu", "cum_bf16.cu",
                              "cum_f64.cu", "cum_i32.cu", "cum_i64.cu"),
}


def kernel_source_hash(workload: str) -> str:
    kind = "cum" if workload.startswith("cum") else "axis" if workload == "axis" else "argreduce"
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "row_wise_arg_gb300", "csrc")
    for n in sorted(_WORKLOAD_SOURCES[kind]):
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(n.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def read_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    src = kernel_source_hash(workload)
    for line in open(p):
        parts = line.split()
        if line.startswith("#") or len(parts) < 3 or parts[0] != workload:
            continue
        return float(parts[1]) if parts[2] == src else None
    return None


def read_config_traffic():
    """Per-case ncu figures of the reduction configs, from the committed
    summary, if taken on the current kernel and planner sources: {case name:
    (DRAM bytes per launch, kernel ns per launch)}."""
    p = os.path.join(ROOT, "profiles", "traffic_configs.txt")
    if not os.path.exists(p):
        return {}
    src = kernel_source_hash("wide_rows")
    out = {}
    for line in open(p):
        parts = line.split()
        if line.startswith("#") or len(parts) < 4:
            continue
        if parts[3] == src:
            out[parts[0]] = (float(parts[1]), float(parts[2]))
    return out


def config_group_cases(groups=range(1, 6)):
    """The reduction configs' cases as the per-config table lists them: the
    duplicated-extreme variants of the wide rows are left out (same shape and
    time as the unique ones)."""
    return [c for g in groups for c in W.config_cases(g) if c.variant != "dup"]


def ncu_cases(torch, A, only: str = None, reps: int = 1):
    """One planner call per reduction config case, in table order, each on
    its own freshly allocated input (for one ncu capture of every case: the
    i-th captured launch is the i-th case printed). `only`: just the cases
    whose name contains it, each called `reps` times (for a full capture of
    one launch, skipping the first); with `only`, the non-last-axis cases are
    searched too."""
    cases = config_group_cases() + (W.config_cases(WORKLOADS["axis"][0]) if only is not None else [])
    for c in cases:
        if only is not None and only not in c.name:
            continue
        x = W.make(c)
        d = to_dev(torch, x, c.dtype)
        out = torch.empty(c.rows * c.inner, dtype=torch.int64, device="cuda")
        for _ in range(reps):
            if c.inner > 1:
                A.argreduce_axis(d.view(c.rows, c.cols, c.inner), 1, c.op, dtype=c.dtype, out_idx=out)
            else:
                A.argreduce(d.view(c.rows, c.cols), c.op, dtype=c.dtype, out_idx=out)
        torch.cuda.synchronize()
        print(c.name, flush=True)
        del d, out


def summarize_ncu(csv_path: str):
    """Turn an ncu CSV of `--ncu-cases` (metrics dram__bytes_read.sum,
    dram__bytes_write.sum, gpu__time_duration.sum) into the lines of
    profiles/traffic_configs.txt: case, bytes, ns, source hash."""
    import csv
    rows = {}
    with open(csv_path) as f:
        lines = [l for l in f if l.startswith('"')]
    for r in csv.DictReader(lines):
        rid = int(r["ID"])
        unit = r.get("Metric Unit", "")
        v = float(r["Metric Value"].replace(",", ""))
        scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9,
                 "nsecond": 1, "usecond": 1e3, "msecond": 1e6, "ns": 1, "us": 1e3, "ms": 1e6}.get(unit, 1)
        rows.setdefault(rid, {})[r["Metric Name"]] = v * scale
    ids = sorted(rows)
    cases = config_group_cases()
    if len(ids) != len(cases):
        raise SystemExit(f"{len(ids)} launches captured for {len(cases)} cases")
    src = kernel_source_hash("wide_rows")
    for c, i in zip(cases, ids):
        m = rows[i]
        b = m["dram__bytes_read.sum"] + m["dram__bytes_write.sum"]
        print(f"{c.name} {b:.0f} {m['gpu__time_duration.sum']:.0f} {src}")


# ---------------------------------------------------------------------------
# Clock sampling during the timed region.
# ---------------------------------------------------------------------------
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) >= 9:
                    rows.append(f)
        except Exception:
            return None
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# Distributed plumbing (replicas: every rank runs the same workload).
# ---------------------------------------------------------------------------
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world <= 1:
        return 0, 1, 0, None
    import torch
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(local)
    dist.init_process_group(backend=backend)
    return rank, world, local, dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device])
        else:
            dist.barrier()


def max_over_ranks(dist, v: float) -> float:
    if dist is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle baseline.
# ---------------------------------------------------------------------------
def oracle_time(cases, inputs, budget_s: float, max_calls: int = None):
    """Time the oracle (as it stands) on host cores over a bounded sample of
    calls, cycling through the cases. Returns (us_per_call, calls, cores)."""
    import oracle
    calls = 0
    cores = 1
    t0 = time.perf_counter()
    while True:
        c = cases[calls % len(cases)]
        if is_scan(c):
            oracle.cumreduce(inputs[calls % len(cases)], c.dtype, c.op, want_val=True)
            used = 1
        elif c.inner > 1:
            oracle.argreduce_axis(inputs[calls % len(cases)], c.dtype, c.op, want_val=False)
            used = 1
        else:
            threads = min(os.cpu_count() or 1, c.rows) if c.rows > 1 else 1
            _, _, used = oracle.argreduce(inputs[calls % len(cases)], c.dtype, c.op, threads=threads,
                                          want_val=False)
        cores = max(cores, used)
        calls += 1
        el = time.perf_counter() - t0
        if (max_calls is not None and calls >= max_calls) or (max_calls is None and el >= budget_s
                                                                and calls >= len(cases)):
            break
    return el * 1e6 / calls, calls, cores, el


# ---------------------------------------------------------------------------
# GPU timing.
# ---------------------------------------------------------------------------
def to_dev(torch, x: np.ndarray, dtype: str):
    view = {"f32": np.float32, "f16": np.int16, "bf16": np.int16, "f64": np.float64, "i32": np.int32,
            "i64": np.int64}[dtype]
    return torch.from_numpy(np.ascontiguousarray(x).view(view)).cuda()


class GraphSet:
    """Calls captured as CUDA graphs over rotating input copies. Graph g runs
    every case once on each of the copies g*per_graph .. (g+1)*per_graph-1,
    so one replay is `per_graph` steps and consecutive uses of a copy are
    separated by all the other copies' bytes."""

    def __init__(self, torch, A, cases, dev_inputs, copies, per_graph, stream, cub=None):
        self.torch = torch
        self.stream = stream
        self.per_graph = per_graph
        self.scratch = A.Scratch()
        need = max([A.argreduce_cum_scratch_bytes(c.rows, c.cols, c.dtype, c.op) if is_scan(c) else
                    A.argreduce_scratch_bytes(c.rows, c.cols, c.dtype, c.op) for c in cases] + [0])
        self.scratch.ensure(max(need, 4096), stream.cuda_stream)
        self.copies = [[x] + [x.clone() for _ in range(copies - 1)] for x in dev_inputs]
        # Scan outputs (an index and a value per element) rotate with the
        # inputs, so that every call writes them to HBM; the reductions'
        # outputs (8 bytes a row) share one buffer per case.
        n_out = [copies if is_scan(c) else 1 for c in cases]
        self.outs = [[torch.empty(max(n_outputs(c), 1), dtype=torch.int64, device="cuda") for _ in range(m)]
                     for c, m in zip(cases, n_out)]
        self.vals = [[torch.empty_like(dev_inputs[i]) for _ in range(n_out[i])] if is_scan(c) else None
                     for i, c in enumerate(cases)]
        self.graphs = []

        def calls(k):
            for i, c in enumerate(cases):
                o = self.outs[i][k % n_out[i]]
                if cub is not None:
                    cub(i, c, self.copies[i][k], o, stream)
                else:
                    call(A, c, self.copies[i][k], o, self.scratch, stream,
                         self.vals[i][k % n_out[i]] if self.vals[i] is not None else None)

        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for k in range(copies):  # eager warm-up of every call
                calls(k)
            stream.synchronize()
            for g0 in range(0, copies, per_graph):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for k in range(g0, g0 + per_graph):
                        calls(k)
                self.graphs.append(g)
        torch.cuda.synchronize()

    def run(self, replays: int, start: int = 0):
        for s in range(replays):
            self.graphs[(start + s) % len(self.graphs)].replay()

    def timed(self, replays: int, warmup: int, dist=None, device=None, clocks=None):
        torch = self.torch
        self.run(warmup)
        torch.cuda.synchronize()
        barrier(dist, device)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if clocks:
            clocks.start()
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            self.run(replays, start=warmup)
            e1.record(self.stream)
        e1.synchronize()
        torch.cuda.synchronize()
        clk = clocks.stop() if clocks else None
        barrier(dist, device)
        return e0.elapsed_time(e1) / 1e3, clk


def copies_for(cases, cap: int = 4096) -> int:
    """Input copies whose total exceeds twice the L2 cache (inputs and, for
    the scan, its per-element outputs)."""
    step_bytes = sum(algo_bytes(c) if is_scan(c) else c.nbytes for c in cases)
    return max(1, min(cap, math.ceil(2 * L2_BYTES / max(step_bytes, 1))))


def time_group(torch, A, cases, inputs, steps, warmup, stream, dist=None, device=None, clocks=None,
               exact: bool = True, cub=None):
    """Time `steps` steps (each: every case once). With exact=True every graph
    is one step (at most 64 copies); otherwise graphs hold several steps and
    the step count is rounded up to whole replays. Returns (seconds, steps
    timed, copies, clocks)."""
    copies = copies_for(cases, cap=64 if exact else 4096)
    if exact:
        per_graph = 1
    else:
        # About 16 calls per graph (as in the timed step) so that a graph
        # launch is not charged to a single call, within 2 GiB of copies.
        step_bytes = sum(algo_bytes(c) if is_scan(c) else c.nbytes for c in cases)
        per_graph = max(1, math.ceil(copies / 16), min(math.ceil(16 / len(cases)), (2 << 30) // max(step_bytes, 1)))
    copies = per_graph * math.ceil(copies / per_graph)
    dev = [to_dev(torch, x, c.dtype).reshape(-1) for c, x in zip(cases, inputs)]
    gs = GraphSet(torch, A, cases, dev, copies, per_graph, stream, cub)
    replays = math.ceil(steps / per_graph)
    secs, clk = gs.timed(replays, max(3, math.ceil(warmup / per_graph)), dist, device, clocks)
    del gs, dev
    return secs, replays * per_graph, copies, clk


def isolated_time(torch, A, c, x, stream, calls: int = 200) -> float:
    """Latency of one call on its own, as a sampler pays it: a sleep kernel
    first holds the stream, so that the host has queued the event, the call
    and the closing event before the GPU reaches them; the median of the
    closing-minus-opening event time over `calls` calls, each on its own
    L2-cold input copy, in microseconds. Unlike the step, no earlier call
    overlaps its launch or its first loads."""
    copies = max(1, min(64, copies_for([c])))
    d0 = to_dev(torch, x, c.dtype).reshape(-1)
    xs = [d0] + [d0.clone() for _ in range(copies - 1)]
    out = torch.empty(max(n_outputs(c), 1), dtype=torch.int64, device="cuda")
    vals = torch.empty_like(d0) if is_scan(c) else None
    scratch = A.Scratch()
    need = (A.argreduce_cum_scratch_bytes(c.rows, c.cols, c.dtype, c.op) if is_scan(c) else
            A.argreduce_scratch_bytes(c.rows, c.cols, c.dtype, c.op))
    scratch.ensure(max(need, 4096), stream.cuda_stream)
    ts = []
    with torch.cuda.stream(stream):
        for k in range(calls + 5):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(100000)  # ~50 us: the host queues what follows meanwhile
            e0.record(stream)
            call(A, c, xs[k % copies], out, scratch, stream, vals)
            e1.record(stream)
            e1.synchronize()
            if k >= 5:
                ts.append(e0.elapsed_time(e1) * 1e3)
    del xs, d0
    return statistics.median(ts)


def cpu_time(c: W.Case, x, budget_s: float = 0.3):
    """The oracle as it stands on one case: all host cores over rows for the
    many-row reductions, one core otherwise; repeated until `budget_s`.
    Returns (us per call, cores)."""
    import oracle
    t0 = time.perf_counter()
    n = 0
    cores = 1
    while True:
        if is_scan(c):
            oracle.cumreduce(x, c.dtype, c.op, want_val=True)
        elif c.inner > 1:
            oracle.argreduce_axis(x, c.dtype, c.op, want_val=False)
        else:
            threads = min(os.cpu_count() or 1, c.rows) if c.rows > 1 else 1
            _, _, cores = oracle.argreduce(x, c.dtype, c.op, threads=threads, want_val=False)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return el * 1e6 / n, cores


def cub_compare(torch, A, cases, inputs, steps, stream, ours_us):
    """cub::DeviceReduce::ArgMax/ArgMin, called as a library, timed exactly as
    the step above (same inputs, copies, graphs and events); its indices are
    first checked against argreduce() on every case."""
    cub = CubCalls(torch, cases)
    agree = True
    for i, (c, x) in enumerate(zip(cases, inputs)):
        d = to_dev(torch, x, c.dtype).reshape(-1)
        mine = torch.empty(1, dtype=torch.int64, device="cuda")
        theirs = torch.empty(1, dtype=torch.int64, device="cuda")
        call(A, c, d, mine, A.Scratch(), stream)
        cub(i, c, d, theirs, stream)
        torch.cuda.synchronize()
        agree = agree and int(mine.item()) == int(theirs.item())
    secs, n, _, _ = time_group(torch, A, cases, inputs, steps, 5, stream, cub=cub)
    us = secs * 1e6 / (n * len(cases))
    return {"impl": "cub::DeviceReduce::ArgMax / ArgMin (CCCL, as a library)", "us_per_call": round(us, 4),
            "argreduce_us_per_call": round(ours_us, 4), "cub_over_argreduce": round(us / ours_us, 3),
            "steps": n, "same_indices": agree,
            "note": "timing comparison only: same inputs, rotating copies, one CUDA graph per copy, CUDA events"}


class E2EStep:
    """One end-to-end step through the public call path with host buffers:
    the step's inputs are copied from one pinned host buffer to the device
    (one copy), the calls run on views of it, and all indices are read back
    into pinned host memory (one copy). Each instance owns its buffers and
    scratch, so two of them can be in flight at once."""

    def __init__(self, torch, A, cases, inputs, host_in, offs):
        view = {"f32": torch.float32, "f16": torch.int16, "bf16": torch.int16, "f64": torch.float64,
                "i32": torch.int32, "i64": torch.int64}
        self.torch, self.A, self.cases = torch, A, cases
        self.host_in = host_in
        self.dev_in = torch.empty(host_in.numel(), dtype=torch.uint8, device="cuda")
        self.devs = [self.dev_in[o:o + c.nbytes].view(view[c.dtype]) for c, o in zip(cases, offs)]
        n_out = [n_outputs(c) for c in cases]
        self.dev_out = torch.empty(sum(n_out), dtype=torch.int64, device="cuda")
        self.outs, k = [], 0
        for n in n_out:
            self.outs.append(self.dev_out[k:k + n])
            k += n
        self.vals = [torch.empty_like(d) if is_scan(c) else None for c, d in zip(cases, self.devs)]
        self.host_out = torch.empty(sum(n_out), dtype=torch.int64).pin_memory()
        self.scratch = A.Scratch()
        need = max([A.argreduce_cum_scratch_bytes(c.rows, c.cols, c.dtype, c.op) if is_scan(c) else
                    A.argreduce_scratch_bytes(c.rows, c.cols, c.dtype, c.op) for c in cases] + [4096])
        self.scratch.ensure(need, torch.cuda.current_stream().cuda_stream)

    def __call__(self, stream):
        self.dev_in.copy_(self.host_in, non_blocking=True)
        for c, d, o, v in zip(self.cases, self.devs, self.outs, self.vals):
            call(self.A, c, d, o, self.scratch, stream, v)
        self.host_out.copy_(self.dev_out, non_blocking=True)


def e2e_time(torch, A, cases, inputs, steps, stream, depth=2):
    """End-to-end steps (E2EStep) captured as `depth` CUDA graphs (each with
    its own buffers) and replayed in rotation on `depth` streams, so up to
    `depth` steps are in flight: later steps' input copies overlap earlier
    steps' calls, as a pipelined application would run them. Also times the
    same steps issued eagerly from Python on one stream (host-bound: the
    binding costs several microseconds a call). Returns (device seconds for
    `steps` pipelined steps, host wall seconds, eager device seconds, h2d, d2h)."""
    offs, total = [], 0
    for c in cases:
        offs.append(total)
        total += -(-c.nbytes // 256) * 256  # every input 256-byte aligned, as an allocator would place it
    host_in = torch.empty(total, dtype=torch.uint8).pin_memory()
    for c, x, o in zip(cases, inputs, offs):
        host_in[o:o + c.nbytes].copy_(torch.from_numpy(np.ascontiguousarray(x).reshape(-1).view(np.uint8)))
    pair = [E2EStep(torch, A, cases, inputs, host_in, offs) for _ in range(depth)]
    h2d = host_in.numel()  # the bytes copied, alignment gaps included
    d2h = pair[0].host_out.numel() * 8
    streams = [stream] + [torch.cuda.Stream() for _ in range(depth - 1)]

    # eager: one step after another on one stream
    with torch.cuda.stream(stream):
        for _ in range(3):
            pair[0](stream)
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            pair[0](stream)
        e1.record(stream)
        e1.synchronize()
        eager = e0.elapsed_time(e1) / 1e3

    graphs = []
    for k in range(depth):
        with torch.cuda.stream(streams[k]):
            pair[k](streams[k])  # warm-up outside the capture
            streams[k].synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=streams[k]):
                pair[k](streams[k])
            graphs.append(g)
    torch.cuda.synchronize()
    for k in range(2 * depth):
        with torch.cuda.stream(streams[k % depth]):
            graphs[k % depth].replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(streams[0])
    for s in streams[1:]:
        s.wait_event(e0)
    for k in range(steps):
        with torch.cuda.stream(streams[k % depth]):
            graphs[k % depth].replay()
    for s in streams[1:]:
        joined = torch.cuda.Event()
        joined.record(s)
        streams[0].wait_event(joined)
    e1.record(streams[0])
    e1.synchronize()
    wall = time.perf_counter() - t0
    return e0.elapsed_time(e1) / 1e3, wall, eager, h2d, d2h


def config_table(torch, A, args, stream, peak):
    """Every workload case (the reductions' configs 1-5 in both tie rules, the
    non-last axis, the scans), timed like the step (graphs of about 16 calls
    on rotating L2-cold inputs), plus for each: its isolated single-call
    latency, the oracle's time on the host cores, and the ncu DRAM figures of
    profiles/traffic_configs.txt where they match the sources. Returns (the
    full table, a compact one of configs 1-5)."""
    table, compact = [], []
    traffic = read_config_traffic()
    for name, (g, _) in sorted(WORKLOADS.items(), key=lambda kv: kv[1][0]):
        if g < 0:
            continue
        gcases = W.config_cases(g)
        ginputs = [W.make(c) for c in gcases]
        for c0, x in zip(gcases, ginputs):
            if c0.variant == "dup":
                continue
            # each case as written, and the same rows with ties to the last index
            variants = [c0] if is_scan(c0) else [c0, dataclasses.replace(c0, op=c0.op + "_last",
                                                                         name=c0.name + "_last")]
            for c in variants:
                n = max(20, min(4000, int(2e9 / max(c.nbytes, 1) / 50)))
                s, n, cp, _ = time_group(torch, A, [c], [x], n, 5, stream, exact=False)
                us = s * 1e6 / n
                gbs = algo_bytes(c) / (s / n) / 1e9
                plan = (A.argreduce_cum_plan(c.rows, c.cols, c.dtype, c.op) if is_scan(c) else
                        A.argreduce_axis_plan(c.rows, c.cols, c.inner, c.dtype, c.op))
                path = plan.as_dict()["path_name"]
                row = {"case": c.name, "us_per_call": round(us, 3), "gbs": round(gbs, 1),
                       "frac": round(gbs / peak, 4), "path": path}
                if c is c0:
                    row["isolated_us"] = round(isolated_time(torch, A, c, x, stream), 3)
                    if not args.no_cpu_baseline:
                        cu, cores = cpu_time(c, x)
                        row["cpu_us_per_call"] = round(cu, 1)
                        row["cpu_cores"] = cores
                    if c.name in traffic:
                        tb, tns = traffic[c.name]
                        row["ncu_dram_bytes"] = int(tb)
                        row["ncu_gbs"] = round(tb / tns, 1)
                        row["ncu_frac"] = round(tb / tns / peak, 4)
                if not args.no_cub and cub_comparable([c]):
                    cs, cn, _, _ = time_group(torch, A, [c], [x], n, 5, stream, exact=False,
                                              cub=CubCalls(torch, [c]))
                    row["cub_us_per_call"] = round(cs * 1e6 / cn, 3)
                if name == "narrow":
                    # the narrow-row target: no slower than a thread-per-row kernel
                    tpr = {}
                    aligned = c.cols * W.ELEM_SIZE[c.dtype] % 16 == 0
                    for label, vec in (("scalar_loads", False), ("vector_loads", True)):
                        if vec and not aligned:
                            continue
                        ts, tn, _, _ = time_group(torch, A, [c], [x], n, 5, stream, exact=False,
                                                  cub=ThreadPerRowCalls(A, [c], vec))
                        tpr[label] = round(ts * 1e6 / tn, 3)
                    row["thread_per_row_us_per_call"] = tpr
                table.append(row)
                if c is c0 and 1 <= g <= 5:
                    # short enough that the last 1500 characters of the line hold every row
                    short = c.name.split("_", 1)[1].replace("_unique", "")
                    frac = f"{row['frac']:.3f}".removeprefix("0")
                    item = f"{short} {row['us_per_call']:.2f} {frac} {path[:2]} i{row['isolated_us']:.1f}"
                    if "cpu_us_per_call" in row:
                        item += f" c{row['cpu_us_per_call']:.0f}/{row['cpu_cores']}"
                    if "ncu_frac" in row:
                        item += " n" + f"{row['ncu_frac']:.3f}".removeprefix("0")
                    compact.append(item)
        del ginputs
    legend = ("case us/call frac-of-HBM-peak path, i: isolated us, c: oracle us/host cores, n: ncu frac")
    return table, {"legend": legend, "rows": compact}


# ---------------------------------------------------------------------------
def reference_arm(args, rank, world, dist):
    """The oracle on host cores, on the same workload and metric."""
    if rank != 0:
        return 0
    group, desc = WORKLOADS[args.workload]
    cases = workload_cases(group)
    inputs = [W.make(c) for c in cases]
    oracle_time(cases, inputs, 0.0, max_calls=min(len(cases), max(1, args.warmup)))
    us, calls, cores, el = oracle_time(cases, inputs, 0.0, max_calls=max(1, args.steps))
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": "us/call", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us * len(cases) / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "+".join(sorted({c.dtype for c in cases})), "data": "synthetic",
        "config": {"workload": args.workload, "description": desc, "cases": len(cases),
                   "step": "one oracle call per step, cycling through the cases (bounded sample)"},
        "cpu_baseline": {"value": us, "unit": "us/call", "cores": cores, "kind": "oracle",
                         "sample": f"{calls} calls cycling over {len(cases)} cases, {el:.2f} s"},
        "e2e": {"value": us, "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="wide_rows", choices=sorted(WORKLOADS))
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload table")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--e2e-depth", type=int, default=3, help="end-to-end steps in flight (graphs in rotation)")
    ap.add_argument("--no-cub", action="store_true", help="skip the cub::DeviceReduce timing comparison")
    ap.add_argument("--ncu-cases", action="store_true",
                    help="no timing: one planner call per reduction config case, for an ncu capture")
    ap.add_argument("--ncu-case", metavar="NAME",
                    help="no timing: three planner calls of each reduction config case (or non-last-axis case) whose name contains NAME")
    ap.add_argument("--ncu-summarize", metavar="CSV",
                    help="no GPU: print profiles/traffic_configs.txt lines from an ncu CSV of --ncu-cases")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.ncu_summarize:
        summarize_ncu(args.ncu_summarize)
        return 0
    if args.ncu_cases or args.ncu_case:
        import torch
        from row_wise_arg_gb300.build import build
        build()
        import row_wise_arg_gb300 as A
        if args.ncu_case:
            ncu_cases(torch, A, only=args.ncu_case, reps=3)
        else:
            ncu_cases(torch, A)
        return 0

    rank, world, local, dist = dist_setup(args.gpus)
    if args.impl == "reference":
        rc = reference_arm(args, rank, world, dist)
        if dist is not None:
            dist.destroy_process_group()
        return rc

    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    from row_wise_arg_gb300.build import build
    if rank == 0 or world == 1:
        build()
    barrier(dist, local if world > 1 else None)
    import row_wise_arg_gb300 as A

    torch.cuda.set_device(local)
    stream = torch.cuda.Stream()
    group, desc = WORKLOADS[args.workload]
    cases = workload_cases(group)
    inputs = [W.make(c) for c in cases]
    step_bytes = sum(algo_bytes(c) for c in cases)
    peak, peak_src = load_peak()

    clocks = Clocks(local)
    secs, _, copies, clk = time_group(torch, A, cases, inputs, args.steps, args.warmup, stream,
                                      dist, local if world > 1 else None, clocks)
    secs = max_over_ranks(dist, secs)
    calls = args.steps * len(cases)
    us_per_call = secs * 1e6 / (calls * world)
    achieved = step_bytes * args.steps / secs / 1e9  # per GPU (every rank runs the same steps)
    plans = {}
    kernels = set()
    for c in cases:
        p = (A.argreduce_cum_plan(c.rows, c.cols, c.dtype, c.op) if is_scan(c) else
             A.argreduce_axis_plan(c.rows, c.cols, c.inner, c.dtype, c.op)).as_dict()
        plans[f"{c.rows}x{c.cols}" + (f"x{c.inner}" if c.inner > 1 else "") + f"_{c.dtype}"] = {k: p[k] for k in ("path_name", "blocks_per_row", "cluster",
                                                                    "block", "unroll", "group", "flags")}
        kernels.add(KERNEL_OF_PATH[p["path_name"]])

    result = {
        "metric": METRIC, "value": round(us_per_call, 4), "unit": "us/call", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs * 1e3 / args.steps, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "+".join(sorted({DTYPE_LABEL[c.dtype] for c in cases})), "data": "synthetic",
        "config": {"workload": args.workload, "description": desc, "calls_per_step": len(cases),
                   "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
                   "l2": f"inputs larger than L2: {copies} rotating copies of the step's inputs "
                         f"({copies * sum(c.nbytes for c in cases) / 2**20:.0f} MiB)",
                   "launch": "CUDA graph per input copy, 16 argreduce calls per graph",
                   "plans": plans},
        "hbm_gbs": round(achieved, 2),
        "gpu_launches": calls,
    }
    result["clocks"] = clk
    traffic = read_traffic(args.workload)
    result["roofline"] = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                          "frac": round(achieved / peak, 5), "traffic": traffic,
                          "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                          else "fallback", "kernel": " + ".join(sorted(kernels)) + " (every call of the step)",
                          "traffic_source": "profiles/traffic.txt (ncu dram__bytes_read.sum + dram__bytes_write.sum "
                                            "per launch, averaged over the step's calls)",
                          "bytes_per_launch_avg": step_bytes / len(cases)}

    if world == 1 or rank == 0:
        dev_s, wall, eager_s, h2d, d2h = e2e_time(torch, A, cases, inputs, args.e2e_steps, stream,
                                                  max(2, args.e2e_depth))
        ncall = args.e2e_steps * len(cases)
        result["e2e"] = {"value": round(dev_s * 1e6 / ncall, 4), "unit": "us/call",
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "host_wall_us_per_call": round(wall * 1e6 / ncall, 4),
                         "eager_python_us_per_call": round(eager_s * 1e6 / ncall, 4),
                         "steps": args.e2e_steps, "steps_in_flight": max(2, args.e2e_depth),
                         "method": "each step copies its inputs from pinned host memory and reads its indices "
                                   "back; steps captured as CUDA graphs (one per step in flight, each with its "
                                   "own buffers) replayed in rotation on as many streams, so later steps' input "
                                   "copies overlap earlier steps' calls"}

    if not args.no_cub and cub_comparable(cases) and (world == 1 or rank == 0):
        result["cub_compare"] = cub_compare(torch, A, cases, inputs, min(args.steps, 4000), stream, us_per_call)

    if not args.no_cpu_baseline and (world == 1 or rank == 0):
        us, ncalls, cores, el = oracle_time(cases, inputs, args.cpu_budget)
        result["cpu_baseline"] = {"value": round(us, 3), "unit": "us/call", "cores": cores, "kind": "oracle",
                                  "sample": f"{ncalls} oracle calls cycling over the {len(cases)} cases of the "
                                            f"step on host cores ({el:.1f} s)"}

    if not args.no_configs and (world == 1 or rank == 0):
        result["configs"], compact = config_table(torch, A, args, stream, peak)
        # printed last, so that the per-config figures of the reduction
        # configs survive a reader that keeps only the end of the line
        result["configs_compact"] = compact

    if world == 1 or rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
