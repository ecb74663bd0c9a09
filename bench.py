"""Benchmark of the same-device collectives on one GB300 (or N replicas).

The timed step is the DTensor redistribution Partial -> Shard(0) ->
Replicate that the DTorch collective-communication page drives through
ConvertKernel::ConvertPlacements (§2.5): a barrier, then ReduceScatter with
kAvg, a barrier, then AllGatherIntoTensor, for P = 4 logical ranks that each
hold a bf16 [8192, 4096] tensor on the same GPU.  The metric is collective
HBM bandwidth: algorithmic bytes (every byte each kernel must read plus every
byte it must write) over device time.

One JSON line on rank 0.  Extra keys: roofline (dominant kernel, measured
here with CUDA events on the launching stream, against the measured HBM copy
peak), cpu_baseline (the CPU oracle on a bounded sample), e2e (the same step
through the public API with pinned host buffers and the copies inside the
timed region), clocks (nvidia-smi during the timed region), gpu_launches, and
rows: one measurement per collective at its own workload (AllReduce P=2 fp32
2^20; bucket all-reduce P=8 of 200 bf16 gradients; AllToAll and uneven
AllGather P=8; barrier latency P=16).

--impl reference times the CPU oracle on a bounded sample of the same workload
instead (the reference arm; there is no other implementation to run).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "collective HBM GB/s (and % of 8 TB/s) per op and size; barrier latency µs"
UNIT = "GB/s"
P_RANKS, ROWS, COLS = 4, 8192, 4096
WORKLOAD = f"rs_avg_then_ag_bf16_P{P_RANKS}_{ROWS}x{COLS}"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["dt_reduce.cu", "dt_copy.cu", "dt_bucket.cu", "dt_barrier.cu", "dt_math.cuh",
                  "dt_internal.h", "dt_device.cuh"]


# ----------------------------------------------------------------- helpers
def step_bytes(P=P_RANKS, rows=ROWS, cols=COLS, es=2):
    n = rows * cols                       # elements per rank
    rs = P * n * es + n * es              # read P full inputs, write P shards (n total)
    ag = n * es + P * n * es              # read P shards, write P full outputs
    return rs, ag


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "of measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "of fallback"


def kernel_source_hash(files=KERNEL_SOURCES):
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(ROOT, "same_device_collective_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, only while the
    sources the kernel is built from (the entry's src_files) are the ones the
    counters were taken on."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[kernel_key]
        if e.get("src_sha") == kernel_source_hash(e.get("src_files", KERNEL_SOURCES)):
            return float(e["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        pass
    return None


class ClockSampler:
    """nvidia-smi samples while the timed region runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self, t0: float, t1: float):
        import datetime
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v == "Active"})
        mhz = sorted(r[1] for r in use)
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(inside),
                "window": "timed region" if inside else "whole run"}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Max over ranks (identity at world size 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(local_ms: float, local_bytes: float, world: int, device=None):
    """Whole-job throughput: bytes of all ranks over the slowest rank's time."""
    ms = reduce_max(local_ms, world, device)
    total = local_bytes * world
    return ms, total / (ms * 1e-3) / 1e9


# ----------------------------------------------------------- CPU oracle leg
def oracle_sample_step(rows_per_rank: int, seed: int = 1):
    """Build a bounded sample of the workload: P ranks of bf16
    [rows_per_rank, COLS], same recipe as the full inputs."""
    from same_device_collective_gb300 import workloads
    import numpy as np
    w = workloads.rs_ag(seed=seed, P=P_RANKS, rows=rows_per_rank, cols=COLS)
    return [x.view(__import__("torch").int16).numpy().view(np.uint16).reshape(-1) for x in w.inputs]


def time_oracle(rows_per_rank: int, min_seconds: float, max_reps: int):
    import oracle
    xs = oracle_sample_step(rows_per_rank)
    rs_b, ag_b = step_bytes(rows=rows_per_rank)
    reps, t0 = 0, time.perf_counter()
    while True:
        rs = oracle.reduce_scatter("bf16", "avg", xs)
        oracle.all_gather(rs)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    return (rs_b + ag_b) * reps / el / 1e9, el, reps


def host_info():
    """The host the CPU baseline ran on: logical CPUs and CPU model."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.TimeoutExpired):
        pass
    import platform
    return {"nproc": os.cpu_count(), "cpu_model": model or platform.machine()}


def time_oracle_configs(min_seconds: float = 1.0):
    """The oracle, single-threaded, on a bounded sample of every other
    configured workload but the RS+AG step (the headline's own sample); GB/s over
    the same algorithmic bytes the GPU rows count."""
    import oracle
    from same_device_collective_gb300 import workloads

    def rate(fn, nbytes):
        fn()
        reps, t0 = 0, time.perf_counter()
        while True:
            fn()
            reps += 1
            el = time.perf_counter() - t0
            if el >= min_seconds:
                return round(nbytes * reps / el / 1e9, 4), reps

    out = {}
    xs = [x.numpy() for x in workloads.allreduce_small().inputs]
    v, reps = rate(lambda: oracle.allreduce("f32", "sum", xs), 2 * 2 * xs[0].size * 4)
    out["allreduce_sum_f32_P2_n2^20"] = {"GB/s": v, "reps": reps, "sample": "the full workload"}

    w = workloads.bucket_grads(T=20)
    grads = [[x.view(__import__("torch").int16).numpy().view(np.uint16) for x in row]
             for row in w.inputs]
    n = sum(w.meta["counts"])
    v, reps = rate(lambda: oracle.bucket_allreduce("bf16", "avg", grads), 2 * 8 * n * 2)
    out["bucket_allreduce_avg_bf16_P8"] = {
        "GB/s": v, "reps": reps,
        "sample": f"20 gradients ({n} bf16 elements per rank) drawn with the 200-tensor recipe"}

    w = workloads.all_to_all_tokens(rows=8192)
    ins = [x.view(__import__("torch").int16).numpy() for x in w.inputs]
    v, reps = rate(lambda: oracle.all_to_all(ins), 2 * 8 * ins[0].size * 2)
    out["all_to_all_bf16_P8"] = {"GB/s": v, "reps": reps,
                                 "sample": "[8192, 4096] per rank (1/8 of the rows)"}

    w = workloads.uneven_gather(max_rows=2048)
    rws = w.meta["rows"]
    ins = [x.numpy() for x in w.inputs]
    v, reps = rate(lambda: oracle.all_gather(ins, rws, 4096 * 4), sum(rws) * 16384 * 9)
    out["uneven_all_gather_i32_P8"] = {"GB/s": v, "reps": reps,
                                       "sample": f"rows {rws} x 4096 (rows up to 2048)"}
    out["sweep_bf16_sum_P4"] = time_oracle_sweep()
    return out


def time_oracle_sweep(P: int = 4, max_bytes: int = 256 << 20, budget_s: float = 45.0):
    """The oracle on the size sweep's inputs (uniform [-1, 1) bf16, seed 4):
    AllReduce and ReduceScatter kSum, AllGather and AllToAll, P = 4, per-rank
    sizes 4 KiB .. 256 MiB (x4), each the median of 3 single calls; GB/s over
    the algorithmic bytes the GPU sweep counts.  Stops early (and says so) past
    budget_s seconds."""
    import oracle
    from same_device_collective_gb300 import workloads
    t_start = time.perf_counter()
    points = {}
    stopped = None
    last = 0.0                                 # seconds the previous size took
    for nbytes in [b for b in workloads.SWEEP_BYTES if b <= max_bytes]:
        spent = time.perf_counter() - t_start
        if spent + 4.5 * last > budget_s:      # the next size moves 4x the bytes
            stopped = f"time budget of {budget_s:.0f} s reached before {nbytes} B per rank"
            break
        t_size = time.perf_counter()
        w = workloads.sweep_inputs(4, P, nbytes, "bf16")
        xs = [x.view(__import__("torch").int16).numpy().view(np.uint16) for x in w.inputs]
        n = xs[0].size
        cases = {
            "allreduce": (lambda: oracle.allreduce("bf16", "sum", xs), 2 * P * nbytes),
            "reduce_scatter": (lambda: oracle.reduce_scatter("bf16", "sum", xs), (P + 1) * nbytes),
            "all_gather": (lambda: oracle.all_gather(xs), (P + P * P) * nbytes),
            "all_to_all": (lambda: oracle.all_to_all(xs), 2 * P * nbytes),
        }
        for op, (fn, b) in cases.items():
            ts = []
            for _ in range(3):
                t0 = time.perf_counter()
                fn()
                ts.append(time.perf_counter() - t0)
            t = sorted(ts)[1]
            points[f"{op}_{nbytes}B"] = {"GB/s": round(b / t / 1e9, 4), "s": round(t, 6)}
        del w, xs
        last = time.perf_counter() - t_size
    return {"points": points, "P": P, "dtype": "bf16", "op": "sum (reductions)",
            "timing": "median of 3 single calls, time.perf_counter", "stopped": stopped}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    rows = 32                                  # [32, 4096] bf16 per rank: 256 KiB
    xs = oracle_sample_step(rows)
    rs_b, ag_b = step_bytes(rows=rows)
    for _ in range(args.warmup):
        oracle.all_gather(oracle.reduce_scatter("bf16", "avg", xs))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.all_gather(oracle.reduce_scatter("bf16", "avg", xs))
    el = time.perf_counter() - t0
    value = (rs_b + ag_b) * args.steps / el / 1e9
    sample = (f"{P_RANKS} ranks x bf16 [{rows}, {COLS}] per step, drawn with the workload's "
              f"recipe (N(0,1), seed 1), single-threaded C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample_rows_per_rank": rows, "P": P_RANKS},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------ GPU arm
STEADY_REPS = 8


def time_events(fn, iters, warmup=3, lead_cycles=4_000_000, reps=1):
    """Median ms per call of fn over iters samples, CUDA events on the current
    stream.  Before each sample the GPU is kept busy (a ~2 ms sleep kernel) so
    that the host has enqueued the sample's work before the start event fires:
    the interval then measures device time, not host marshalling.  A sample is
    `reps` back-to-back calls and reports their mean: with reps > 1 every call
    but the first also pays for writing back the dirty L2 lines its
    predecessor left, as calls in a loop do (steady state)."""
    import torch
    for _ in range(warmup):
        fn()
    st = [torch.cuda.Event(enable_timing=True) for _ in range(iters)]
    en = [torch.cuda.Event(enable_timing=True) for _ in range(iters)]
    torch.cuda.synchronize()
    for i in range(iters):
        torch.cuda._sleep(lead_cycles)
        st[i].record()
        for _ in range(reps):
            fn()
        en[i].record()
    torch.cuda.synchronize()
    ts = sorted(s.elapsed_time(e) / reps for s, e in zip(st, en))
    return ts[len(ts) // 2]


ROW_NAMES = ["allreduce_small", "allreduce_large", "bucket", "all_to_all", "uneven_all_gather",
             "barrier", "rank_local", "placements", "hsdp_pipeline", "sweep_points", "misaligned"]


class HsdpSchedule:
    """The hyper-parallel post_backward schedule on a 2 x 2 mesh of logical
    ranks (two shard groups, two replicate groups), 8 modules of bf16
    gradients (32 Mi elements per rank per module); each module's backward
    compute is stood in for by a bf16 GEMM on the compute stream.  sequential:
    compute, ReduceScatter, AllReduce per module on one stream; pipelined: the
    same work with the collectives in async scopes on the groups' own streams
    (wait previous RS, issue RS, issue previous AR).  `mark`, when given, is
    called with (stream, tag) before (tag 2m) and after (2m + 1) module m's
    GEMM."""

    def __init__(self, dt, dev, M=8, n=32 << 20):
        import torch
        self.dt, self.M, self.n = dt, M, n
        gen = torch.Generator(device=dev).manual_seed(7)
        self.grads = [[torch.randn(n, generator=gen, device=dev).to(torch.bfloat16) for _ in range(4)]
                      for _ in range(M)]
        self.rsb = [[torch.empty(n // 2, dtype=torch.bfloat16, device=dev) for _ in range(4)]
                    for _ in range(M)]
        self.fin = [[torch.empty(n // 2, dtype=torch.bfloat16, device=dev) for _ in range(4)]
                    for _ in range(M)]
        self.a = torch.randn(8192, 8192, generator=gen, device=dev).to(torch.bfloat16)
        self.b = torch.randn(8192, 4096, generator=gen, device=dev).to(torch.bfloat16)
        self.c = torch.empty(8192, 4096, dtype=torch.bfloat16, device=dev)
        self.shard = [dt.dt_group_create(2, dev.index) for _ in range(2)]
        self.repl = [dt.dt_group_create(2, dev.index) for _ in range(2)]
        self.compute = torch.cuda.Stream(dev)
        self.craw = self.compute.cuda_stream
        self.comm_bytes = M * 2 * ((2 + 1) * n * 2 + 2 * 2 * (n // 2) * 2)
        self.mark = None

    def gemm(self, m):
        import torch
        if self.mark:
            self.mark(self.craw, 2 * m)
        torch.matmul(self.a, self.b, out=self.c)
        if self.mark:
            self.mark(self.craw, 2 * m + 1)

    def rs_of(self, m, stream):
        for s_ in range(2):
            self.rs_of_one(m, s_, stream)

    def ar_of(self, m, stream):
        for k in range(2):
            self.ar_of_one(m, k, stream)

    def gemm_only(self):
        import torch
        with torch.cuda.stream(self.compute):
            for m in range(self.M):
                self.gemm(m)

    def sequential(self):
        import torch
        with torch.cuda.stream(self.compute):
            for m in range(self.M):
                self.gemm(m)
                self.rs_of(m, self.craw)
                self.ar_of(m, self.craw)

    def pipelined(self):
        import torch
        dt = self.dt
        with torch.cuda.stream(self.compute):
            prev, pend = [], []
            for m in range(self.M):
                self.gemm(m)                                   # module m's backward
                for w_ in prev:
                    dt.dt_work_wait(w_, self.compute)
                    dt.dt_work_free(w_)
                cur = []
                for s_ in range(2):
                    cs = dt.dt_async_begin(self.shard[s_], self.compute)
                    self.rs_of_one(m, s_, cs)
                    cur.append(dt.dt_async_end(self.shard[s_]))
                if m > 0:
                    for k in range(2):
                        cs = dt.dt_async_begin(self.repl[k], self.compute)
                        self.ar_of_one(m - 1, k, cs)
                        pend.append(dt.dt_async_end(self.repl[k]))
                prev = cur
            for w_ in prev:
                dt.dt_work_wait(w_, self.compute)
                dt.dt_work_free(w_)
            for k in range(2):
                cs = dt.dt_async_begin(self.repl[k], self.compute)
                self.ar_of_one(self.M - 1, k, cs)
                pend.append(dt.dt_async_end(self.repl[k]))
            for w_ in pend:
                dt.dt_work_wait(w_, self.compute)
                dt.dt_work_free(w_)

    def rs_of_one(self, m, s_, stream):
        dt, n = self.dt, self.n
        x, y = 2 * s_, 2 * s_ + 1
        dt.dt_reduce_scatter(self.shard[s_], dt.DT_ALL_RANKS, [self.grads[m][x], self.grads[m][y]],
                             [self.rsb[m][x], self.rsb[m][y]], n // 2, "bf16", "avg", stream)

    def ar_of_one(self, m, k, stream):
        dt, n = self.dt, self.n
        dt.dt_allreduce(self.repl[k], dt.DT_ALL_RANKS, [self.rsb[m][k], self.rsb[m][k + 2]],
                        [self.fin[m][k], self.fin[m][k + 2]], n // 2, "bf16", "avg", 0, stream)

    def close(self):
        import torch
        torch.cuda.synchronize()
        ok = all(self.dt.dt_group_check(x) == self.dt.DT_OK for x in self.shard + self.repl)
        for x in self.shard + self.repl:
            self.dt.dt_group_destroy(x)
        return ok


def measure_rows(dt, dev, peak, only=None):
    """One measurement per collective at its own workload (device-resident).
    `only` restricts it to one of ROW_NAMES."""
    import torch
    from same_device_collective_gb300 import workloads
    rows = {}
    ALL = dt.DT_ALL_RANKS

    def rec(name, nbytes, ms, **extra):
        gbs = nbytes / (ms * 1e-3) / 1e9
        rows[name] = {"GB/s": round(gbs, 1), "us": round(ms * 1e3, 2), "bytes": nbytes,
                      "frac_of_measured_hbm": round(gbs / peak, 4),
                      "frac_of_8TBs": round(gbs / NOMINAL_HBM_GBS, 4), **extra}

    def want(name):
        return only is None or only == name

    # A1: AllReduce kSum, P=2, fp32 2^20 per rank (16 MiB moved: L2-resident,
    # launch-bound): per-call device time from a replayed CUDA graph of 100
    # calls, and per call when issued one by one from Python
    if want("allreduce_small"):
        w = workloads.allreduce_small()
        xs = [x.to(dev) for x in w.inputs]
        outs = [torch.empty_like(x) for x in xs]
        g = dt.dt_group_create(2, dev.index)
        n = xs[0].numel()
        ms_stream = time_events(lambda: dt.dt_allreduce(g, ALL, xs, outs, n, "f32", "sum"), 200)
        ms_graph = None
        try:
            st = torch.cuda.Stream(dev)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(st):
                with torch.cuda.graph(graph, stream=st):
                    for _ in range(100):
                        dt.dt_allreduce(g, ALL, xs, outs, n, "f32", "sum", 0, st)
            graph.replay()
            torch.cuda.synchronize()
            ms_graph = time_events(graph.replay, 20) / 100
        except Exception:
            ms_graph = None
        rec("allreduce_sum_f32_P2_n2^20", 2 * 2 * n * 4, ms_graph if ms_graph else ms_stream,
            l2_resident=True, timing="CUDA graph of 100 calls" if ms_graph else "per call",
            us_per_call_issued_from_python=round(ms_stream * 1e3, 2))
        dt.dt_group_destroy(g)
        del xs, outs

    # A1 at bandwidth scale: AllReduce kSum P=8 fp32, 64 MiB per rank
    if want("allreduce_large"):
        n = 16 << 20
        gen = torch.Generator(device=dev).manual_seed(4)
        xs = [torch.rand(n, generator=gen, device=dev) for _ in range(8)]
        outs = [torch.empty_like(x) for x in xs]
        g = dt.dt_group_create(8, dev.index)
        ms = time_events(lambda: dt.dt_allreduce(g, ALL, xs, outs, n, "f32", "sum"), 20,
                         reps=STEADY_REPS)
        rec("allreduce_sum_f32_P8_64MiB", 2 * 8 * n * 4, ms)
        dt.dt_group_destroy(g)
        del xs, outs

    # A5: fused bucket all-reduce kAvg, P=8, 200 bf16 gradients, 25 MiB buckets
    if want("bucket"):
        w = workloads.bucket_grads(device=str(dev))
        counts = w.meta["counts"]
        g = dt.dt_group_create(8, dev.index)
        _, nb = dt.dt_bucket_plan(counts, 2, workloads.BUCKET_CAP_BYTES)
        # gradients stay allocated across steps: their pointer table is built once
        table, cnt = dt.pointer_table(w.inputs), np.asarray(counts, dtype=np.uint64)
        ms = time_events(lambda: dt.dt_bucket_allreduce(g, table, cnt, "bf16", "avg",
                                                        workloads.BUCKET_CAP_BYTES), 20,
                         reps=STEADY_REPS)
        rec("bucket_allreduce_avg_bf16_P8_T200", 2 * 8 * sum(counts) * 2, ms, buckets=nb,
            barriers=nb - 1)
        dt.dt_group_destroy(g)
        # the allocation-free entry point on the same gradients: device time,
        # and the host time of one call when it copies its tables (stream idle)
        # and when it repeats the previous call's tables
        cap = workloads.BUCKET_CAP_BYTES
        static = lambda c=cap: dt.dt_bucket_allreduce_static(8, table, cnt, "bf16", "avg", c)
        ms = time_events(static, 20, reps=STEADY_REPS)
        copy_us, reuse_us = [], []
        for i in range(20):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            static(cap - 4096 * (i % 2))           # other buckets than the call before
            copy_us.append((time.perf_counter() - t0) * 1e6)
        torch.cuda.synchronize()
        static()
        for _ in range(50):
            t0 = time.perf_counter()
            static()
            reuse_us.append((time.perf_counter() - t0) * 1e6)
        torch.cuda.synchronize()
        rec("bucket_allreduce_static_avg_bf16_P8_T200", 2 * 8 * sum(counts) * 2, ms, buckets=nb,
            barriers=0, host_us_tables_copied=round(sorted(copy_us)[len(copy_us) // 2], 1),
            host_us_tables_reused=round(sorted(reuse_us)[len(reuse_us) // 2], 1),
            note="no group: stream order between buckets, no signal barrier")
        del w

    # A4: AllToAll P=8, bf16 [65536, 4096] per rank
    if want("all_to_all"):
        w = workloads.all_to_all_tokens(device=str(dev))
        outs = [torch.empty_like(x) for x in w.inputs]
        g = dt.dt_group_create(8, dev.index)
        nbytes_rank = w.inputs[0].numel() * 2
        ms = time_events(lambda: dt.dt_all_to_all(g, ALL, w.inputs, outs, nbytes_rank // 8), 10,
                         reps=STEADY_REPS)
        rec("all_to_all_bf16_P8_65536x4096", 2 * 8 * nbytes_rank, ms)
        dt.dt_group_destroy(g)
        del w, outs

    # A3b: uneven AllGather P=8, int32 rows U[1,16384] x 4096 (per-rank outputs)
    if want("uneven_all_gather"):
        w = workloads.uneven_gather(device=str(dev))
        rws = w.meta["rows"]
        total = sum(rws)
        outs = [torch.empty(total, 4096, dtype=torch.int32, device=dev) for _ in range(8)]
        g = dt.dt_group_create(8, dev.index)
        ms = time_events(lambda: dt.dt_all_gather(g, ALL, w.inputs, outs, rws, 0, 4096 * 4), 10,
                         reps=STEADY_REPS)
        rec("uneven_all_gather_i32_P8", total * 16384 * (1 + 8), ms, rows=rws)
        dt.dt_group_destroy(g)
        del outs
        shared = torch.empty(total, 4096, dtype=torch.int32, device=dev)
        g = dt.dt_group_create(8, dev.index)
        ms = time_events(lambda: dt.dt_all_gather(g, ALL, w.inputs, [shared] * 8, rws, 0, 4096 * 4,
                                                  flags=dt.DT_SHARED_OUTPUT), 10, reps=STEADY_REPS)
        rec("uneven_all_gather_i32_P8_shared_output", total * 16384 * 2, ms)
        dt.dt_group_destroy(g)
        del w, shared

    # A6: barrier latency, P=16, 10^5 back-to-back calls (and as a replayed CUDA graph)
    if want("barrier"):
        g = dt.dt_group_create(16, dev.index)
        calls = 100_000
        for _ in range(100):
            dt.dt_barrier(g)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        raw = torch.cuda.current_stream(dev).cuda_stream
        s.record()
        for _ in range(calls):
            dt.dt_barrier(g, ALL, raw)
        e.record()
        torch.cuda.synchronize()
        us_direct = s.elapsed_time(e) * 1e3 / calls
        bar = dt.prepare(dt.dt_barrier, g, ALL, raw)     # the same call, marshalled once
        s.record()
        for _ in range(calls):
            bar()
        e.record()
        torch.cuda.synchronize()
        us_prepared = s.elapsed_time(e) * 1e3 / calls
        us_graph = None
        try:
            stream = torch.cuda.Stream(dev)
            per_graph = 1000
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(graph, stream=stream):
                    for _ in range(per_graph):
                        dt.dt_barrier(g, stream=stream)
            torch.cuda.synchronize()
            graph.replay()
            torch.cuda.synchronize()
            s.record()
            for _ in range(calls // per_graph):
                graph.replay()
            e.record()
            torch.cuda.synchronize()
            us_graph = s.elapsed_time(e) * 1e3 / calls
        except Exception as ex:   # capture support is reported, not required
            us_graph = f"capture failed: {type(ex).__name__}"
        win_ok = dt.dt_group_check(g) == dt.DT_OK
        dt.dt_group_destroy(g)
        rows["barrier_P16"] = {"us_per_call_stream": round(us_direct, 3),
                               "us_per_call_stream_prepared": round(us_prepared, 3),
                               "us_per_call_graph": us_graph if isinstance(us_graph, str)
                               else round(us_graph, 3), "calls": calls, "status_ok": win_ok}

    # Rank-local mode: four host threads, one per rank, each with its own
    # stream, drive the configured RS(avg) + AG step (barrier, RS, barrier,
    # AG); every call meets on the host and the last rank launches.  Wall time
    # of K steps after both ends are synchronised.
    if want("rank_local"):
        import threading
        P, R, C = P_RANKS, ROWS, COLS
        w = workloads.rs_ag(seed=1, P=P, rows=R, cols=C, device=str(dev))
        xs = w.inputs
        m = R // P * C
        rs = [torch.empty(R // P, C, dtype=torch.bfloat16, device=dev) for _ in range(P)]
        ag = [torch.empty(R, C, dtype=torch.bfloat16, device=dev) for _ in range(P)]
        streams = [torch.cuda.Stream(dev) for _ in range(P)]
        raws = [s_.cuda_stream for s_ in streams]
        g = dt.dt_group_create(P, dev.index)

        # each rank's four calls, marshalled once (dt.prepare)
        prepared = [[dt.prepare(dt.dt_barrier, g, r, raws[r]),
                     dt.prepare(dt.dt_reduce_scatter, g, r, [xs[r]], [rs[r]], m, "bf16", "avg",
                                raws[r]),
                     dt.prepare(dt.dt_barrier, g, r, raws[r]),
                     dt.prepare(dt.dt_all_gather, g, r, [rs[r]], [ag[r]], None, R // P, C * 2, 0,
                                raws[r])] for r in range(P)]

        def rank_steps_prepared(r, k):
            torch.cuda.set_device(dev)
            calls = prepared[r]
            for _ in range(k):
                for c in calls:
                    c()

        def rank_steps(r, k):
            torch.cuda.set_device(dev)
            for _ in range(k):
                dt.dt_barrier(g, r, raws[r])
                dt.dt_reduce_scatter(g, r, [xs[r]], [rs[r]], m, "bf16", "avg", raws[r])
                dt.dt_barrier(g, r, raws[r])
                dt.dt_all_gather(g, r, [rs[r]], [ag[r]], None, R // P, C * 2, 0, raws[r])

        def run(body, k):
            ts = [threading.Thread(target=body, args=(r, k)) for r in range(P)]
            for t in ts:
                t.start()
            for t in ts:
                t.join()

        K = 500
        rs_b, ag_b = step_bytes()
        timing = {}
        for name, body in (("prepared", rank_steps_prepared), ("per_call", rank_steps)):
            run(body, 20)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            run(body, K)
            torch.cuda.synchronize()
            timing[name] = time.perf_counter() - t0
        el = timing["prepared"]
        gbs = (rs_b + ag_b) * K / el / 1e9
        ok = dt.dt_group_check(g) == dt.DT_OK
        dt.dt_group_destroy(g)
        rows["rank_local_rs_ag_step_bf16_P4"] = {
            "GB/s": round(gbs, 1), "us_per_step": round(el / K * 1e6, 2), "steps": K,
            "frac_of_measured_hbm": round(gbs / peak, 4), "threads": P, "status_ok": ok,
            "timing": "wall clock over K steps, both ends synchronised",
            "caller": "Python threads, prepared calls (arguments marshalled once)",
            "per_call_functions": {
                "us_per_step": round(timing["per_call"] / K * 1e6, 2),
                "GB/s": round((rs_b + ag_b) * K / timing["per_call"] / 1e9, 1),
                "note": "arguments marshalled on every call, under the interpreter lock"}}
        del w, xs, rs, ag
        torch.cuda.synchronize()
        # the same step from native threads: the library's own rank-local cost
        tool = os.path.join(ROOT, "same_device_collective_gb300", "rank_local_step")
        try:
            res = subprocess.run([tool, str(P), str(R), str(C), "2000"], capture_output=True,
                                 text=True, timeout=300)
            native = json.loads(res.stdout.strip().splitlines()[-1])
            if "GB/s" in native:
                native["frac_of_measured_hbm"] = round(native["GB/s"] / peak, 4)
            native["caller"] = "C++ std::thread per rank (rank_local_step)"
        except (OSError, ValueError, IndexError, subprocess.TimeoutExpired) as ex:
            native = {"error": f"{type(ex).__name__}: {ex}"}
        rows["rank_local_rs_ag_step_bf16_P4_native_threads"] = native
        # the same with one stream shared by all rank threads: no cross-stream
        # event waits, so the gap to the row above is what those waits cost
        try:
            res = subprocess.run([tool, str(P), str(R), str(C), "2000", "shared"], capture_output=True,
                                 text=True, timeout=300)
            shared = json.loads(res.stdout.strip().splitlines()[-1])
            if "GB/s" in shared:
                shared["frac_of_measured_hbm"] = round(shared["GB/s"] / peak, 4)
            shared["caller"] = "C++ std::thread per rank (rank_local_step), one shared stream"
        except (OSError, ValueError, IndexError, subprocess.TimeoutExpired) as ex:
            shared = {"error": f"{type(ex).__name__}: {ex}"}
        rows["rank_local_rs_ag_step_bf16_P4_native_threads_shared_stream"] = shared

    # Remaining placement conversions at the configured shapes: R -> S of a
    # replicated bf16 [8192, 4096] tensor (P=4), AllGatherIntoVec of its
    # shards, S(0) -> S(1) AllToAll of P=8 bf16 [65536, 4096] token matrices,
    # and the page-literal stepwise bf16 sum as a ReduceScatter (P=4).
    if want("placements"):
        P, R, C = P_RANKS, ROWS, COLS
        gen = torch.Generator(device=dev).manual_seed(1)
        full = [torch.randn(R, C, generator=gen, device=dev).to(torch.bfloat16) for _ in range(P)]
        shards = [torch.empty(R // P, C, dtype=torch.bfloat16, device=dev) for _ in range(P)]
        g = dt.dt_group_create(P, dev.index)
        ms = time_events(lambda: dt.dt_replicate_to_shard(g, ALL, full, shards, None, R, C * 2), 20,
                         reps=STEADY_REPS)
        rec("replicate_to_shard_bf16_P4_8192x4096", 2 * R * C * 2, ms)
        vec = [torch.empty(R // P, C, dtype=torch.bfloat16, device=dev) for _ in range(P * P)]
        ms = time_events(lambda: dt.dt_all_gather_into_vec(g, ALL, shards, vec, None, R // P, C * 2),
                         20, reps=STEADY_REPS)
        rec("all_gather_into_vec_bf16_P4_2048x4096", (P + P * P) * (R // P) * C * 2, ms)
        del vec
        # the plain AllGather of the same shards, timed the same way (in the
        # bench step it reads its input from L2; here, as above, from HBM)
        ag = [torch.empty(R, C, dtype=torch.bfloat16, device=dev) for _ in range(P)]
        ms = time_events(lambda: dt.dt_all_gather(g, ALL, shards, ag, None, R // P, C * 2), 20,
                         reps=STEADY_REPS)
        rec("all_gather_bf16_P4_2048x4096", (P + P * P) * (R // P) * C * 2, ms)
        del ag
        rsb = [torch.empty(R // P, C, dtype=torch.bfloat16, device=dev) for _ in range(P)]
        ms = time_events(lambda: dt.dt_reduce_scatter(g, ALL, full, rsb, R // P * C, "bf16",
                                                      "sum_stepwise"), 20, reps=STEADY_REPS)
        rec("reduce_scatter_sum_stepwise_bf16_P4_8192x4096", (P + 1) * R * C * 2, ms)
        dt.dt_group_destroy(g)
        del full, shards, rsb
        w = workloads.all_to_all_tokens(device=str(dev))
        R8, C8 = w.inputs[0].shape
        outs = [torch.empty(8 * R8, C8 // 8, dtype=torch.bfloat16, device=dev) for _ in range(8)]
        g = dt.dt_group_create(8, dev.index)
        ms = time_events(lambda: dt.dt_all_to_all_2d(g, ALL, w.inputs, outs, R8, C8, 2, 0, 1), 10,
                         reps=STEADY_REPS)
        rec("all_to_all_S0_to_S1_bf16_P8_65536x4096", 2 * 8 * R8 * C8 * 2, ms)
        dt.dt_group_destroy(g)
        del w, outs

    # Async works: the hyper-parallel post_backward schedule on a 2 x 2 mesh of
    # logical ranks (two shard groups, two replicate groups), 8 modules of
    # bf16 gradients (32 Mi elements per rank per module); each module's
    # backward compute is stood in for by a bf16 GEMM on the compute stream.
    # Sequential: compute, ReduceScatter, AllReduce per module on one stream.
    # Pipelined: the same work with the collectives in async scopes on the
    # groups' own streams (wait previous RS, issue RS, issue previous AR).
    if want("hsdp_pipeline"):
        h = HsdpSchedule(dt, dev)

        def wall(fn, reps=5):
            fn()
            torch.cuda.synchronize()
            ts = []
            for _ in range(reps):
                t0 = time.perf_counter()
                fn()
                torch.cuda.synchronize()
                ts.append(time.perf_counter() - t0)
            return sorted(ts)[reps // 2]

        t_gemm = wall(h.gemm_only)
        t_seq = wall(h.sequential)
        t_pipe = wall(h.pipelined)
        ok = h.close()
        rows["hsdp_pipeline_2x2_bf16_M8"] = {
            "us_sequential": round(t_seq * 1e6, 1), "us_pipelined": round(t_pipe * 1e6, 1),
            "us_compute_only": round(t_gemm * 1e6, 1),
            "speedup": round(t_seq / t_pipe, 3),
            "comm_GB/s_sequential_excl_compute": round(h.comm_bytes / max(t_seq - t_gemm, 1e-9) / 1e9, 1),
            "status_ok": ok, "timing": "wall clock, median of 5, synchronised"}
        del h

    # Size sweep (config 5) at the message sizes the HBM target is stated
    # for: every op at P = 2 and P = 16, bf16 kSum, 64 MiB and 256 MiB per
    # rank, per-rank outputs; seeded uniform [-1, 1) inputs drawn on the
    # device.  Timed like the other rows (8 back-to-back calls per sample).
    if want("sweep_points"):
        torch.cuda.empty_cache()
        points = {}
        for P in (2, 16):
            g = dt.dt_group_create(P, dev.index)
            for nbytes in (64 << 20, 256 << 20):
                gen = torch.Generator(device=dev).manual_seed(4)
                n = nbytes // 2
                xs = [(torch.rand(n, generator=gen, device=dev) * 2 - 1).to(torch.bfloat16)
                      for _ in range(P)]
                outs = [torch.empty_like(x) for x in xs]
                res = {}
                ms = time_events(lambda: dt.dt_allreduce(g, ALL, xs, outs, n, "bf16", "sum"), 5,
                                 reps=STEADY_REPS)
                res["allreduce"] = (2 * P * nbytes, ms)
                rs = [torch.empty(n // P, dtype=torch.bfloat16, device=dev) for _ in range(P)]
                ms = time_events(lambda: dt.dt_reduce_scatter(g, ALL, xs, rs, n // P, "bf16", "sum"), 5,
                                 reps=STEADY_REPS)
                res["reduce_scatter"] = ((P + 1) * nbytes, ms)
                del rs
                ms = time_events(lambda: dt.dt_all_to_all(g, ALL, xs, outs, nbytes // P), 5,
                                 reps=STEADY_REPS)
                res["all_to_all"] = (2 * P * nbytes, ms)
                del outs
                ag = [torch.empty(P * n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
                ms = time_events(lambda: dt.dt_all_gather(g, ALL, xs, ag, None, 1, nbytes), 5,
                                 reps=STEADY_REPS)
                res["all_gather"] = ((P + P * P) * nbytes, ms)
                del ag, xs
                torch.cuda.empty_cache()
                for op, (b, t) in res.items():
                    gbs = b / (t * 1e-3) / 1e9
                    points[f"{op}_P{P}_{nbytes >> 20}MiB"] = {
                        "GB/s": round(gbs, 1), "us": round(t * 1e3, 2),
                        "frac_of_8TBs": round(gbs / NOMINAL_HBM_GBS, 4),
                        "frac_of_measured_hbm": round(gbs / peak, 4)}
            assert dt.dt_group_check(g) == dt.DT_OK
            dt.dt_group_destroy(g)
        fr = [v["frac_of_8TBs"] for v in points.values()]
        rows["sweep_points_bf16_sum_P2_P16_64_256MiB"] = {
            "points": points, "min_frac_of_8TBs": min(fr),
            "points_at_or_above_0.80": sum(f >= 0.8 for f in fr), "n_points": len(fr),
            "outputs": "per-rank", "inputs": "uniform [-1, 1) bf16, seed 4, drawn on the device"}

    # Buffers off a 16-byte boundary.  The configured RS(avg) + AG step on
    # bf16 views that all start 2 bytes past a boundary (every buffer shares
    # the offset: the vector kernels run from each buffer's first boundary),
    # against the same step on aligned buffers; and an AllGather whose shards
    # start 2 bytes past a boundary while the outputs are aligned (sources and
    # destinations at different offsets: the shifting copy).
    if want("misaligned"):
        P, R, C = P_RANKS, ROWS, COLS
        gen = torch.Generator(device=dev).manual_seed(1)
        m = R // P * C

        def views(nelem, off_bytes, k):
            base = [torch.empty(nelem + 16, dtype=torch.bfloat16, device=dev) for _ in range(k)]
            return base, [b_[off_bytes // 2:off_bytes // 2 + nelem] for b_ in base]

        res = {}
        for name, off in (("aligned", 0), ("views_2B_past_boundary", 2)):
            _, xs = views(R * C, off, P)
            for x in xs:
                x.copy_(torch.randn(R * C, generator=gen, device=dev).to(torch.bfloat16))
            _, rs = views(m, off, P)
            _, ag = views(R * C, off, P)
            g = dt.dt_group_create(P, dev.index)

            def step():
                dt.dt_barrier(g)
                dt.dt_reduce_scatter(g, ALL, xs, rs, m, "bf16", "avg")
                dt.dt_barrier(g)
                dt.dt_all_gather(g, ALL, rs, ag, None, R // P, C * 2)

            ms = time_events(step, 20, reps=STEADY_REPS)
            ok = dt.dt_group_check(g) == dt.DT_OK
            dt.dt_group_destroy(g)
            res[name] = (ms, ok)
            del xs, rs, ag
        rs_b, ag_b = step_bytes()
        ms0, ms1 = res["aligned"][0], res["views_2B_past_boundary"][0]
        rows["rs_ag_step_bf16_P4_views_2B_past_boundary"] = {
            "GB/s": round((rs_b + ag_b) / (ms1 * 1e-3) / 1e9, 1), "us": round(ms1 * 1e3, 2),
            "aligned_us": round(ms0 * 1e3, 2), "ratio_to_aligned": round(ms0 / ms1, 4),
            "status_ok": res["aligned"][1] and res["views_2B_past_boundary"][1]}
        # the shifting copy: shards 2 bytes past a boundary, aligned outputs
        n = 32 << 20                              # 64 MiB of bf16 per shard
        g = dt.dt_group_create(P, dev.index)
        res = {}
        for name, off in (("aligned", 0), ("shards_2B_past_boundary", 2)):
            _, sh = views(n, off, P)
            for x in sh:
                x.copy_(torch.rand(n, generator=gen, device=dev).to(torch.bfloat16))
            ag = [torch.empty(P * n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
            res[name] = time_events(lambda: dt.dt_all_gather(g, ALL, sh, ag, None, 1, n * 2), 10,
                                    reps=STEADY_REPS)
            del sh, ag
        ok = dt.dt_group_check(g) == dt.DT_OK
        dt.dt_group_destroy(g)
        b = (P + P * P) * n * 2
        ms0, ms1 = res["aligned"], res["shards_2B_past_boundary"]
        rows["all_gather_bf16_P4_64MiB_shards_2B_past_boundary"] = {
            "GB/s": round(b / (ms1 * 1e-3) / 1e9, 1), "us": round(ms1 * 1e3, 2),
            "aligned_us": round(ms0 * 1e3, 2), "ratio_to_aligned": round(ms0 / ms1, 4),
            "status_ok": ok}
        # an AllReduce whose inputs start 0, 2, 4, 6 bytes past a boundary
        # (aligned outputs: the shifting reduction), beside the aligned call
        n = 32 << 20                              # 64 MiB of bf16 per rank
        g = dt.dt_group_create(P, dev.index)
        res = {}
        for name, offs in (("aligned", (0, 0, 0, 0)), ("inputs_at_own_offsets", (0, 2, 4, 6))):
            base = [torch.empty(n + 8, dtype=torch.bfloat16, device=dev) for _ in range(P)]
            xs = [b_[o // 2:o // 2 + n] for b_, o in zip(base, offs)]
            for x in xs:
                x.copy_(torch.rand(n, generator=gen, device=dev).to(torch.bfloat16))
            outs = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
            res[name] = time_events(lambda: dt.dt_allreduce(g, ALL, xs, outs, n, "bf16", "sum"), 10,
                                    reps=STEADY_REPS)
            del base, xs, outs
        ok = dt.dt_group_check(g) == dt.DT_OK
        dt.dt_group_destroy(g)
        b = 2 * P * n * 2
        ms0, ms1 = res["aligned"], res["inputs_at_own_offsets"]
        rows["allreduce_bf16_P4_64MiB_inputs_at_own_offsets"] = {
            "GB/s": round(b / (ms1 * 1e-3) / 1e9, 1), "us": round(ms1 * 1e3, 2),
            "aligned_us": round(ms0 * 1e3, 2), "ratio_to_aligned": round(ms0 / ms1, 4),
            "status_ok": ok}

    torch.cuda.empty_cache()
    return rows


def run_e2e(dt, g, xs, P, rows_, cols, m, steps, world, dev):
    """Pipelined end-to-end steps; returns (ms, GB/s, h2d bytes, d2h bytes)."""
    import torch
    ALL = dt.DT_ALL_RANKS
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    h_in = [x.cpu().pin_memory() for x in xs]
    sets = []
    for _ in range(2):
        sets.append({
            "in": [torch.empty_like(x) for x in xs],
            "rs": [torch.empty(rows_ // P, cols, dtype=torch.bfloat16, device=dev) for _ in range(P)],
            "ag": [torch.empty(rows_, cols, dtype=torch.bfloat16, device=dev) for _ in range(P)],
            "h_out": [torch.empty(rows_, cols, dtype=torch.bfloat16).pin_memory() for _ in range(P)],
            "ev_in": torch.cuda.Event(), "ev_done": torch.cuda.Event(), "ev_out": torch.cuda.Event(),
        })
    raw = comp.cuda_stream

    def one(i):
        st = sets[i % 2]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(st["ev_done"])          # step i-2 is done reading this set
            for d, h in zip(st["in"], h_in):
                d.copy_(h, non_blocking=True)
            st["ev_in"].record(s_in)
        comp.wait_event(st["ev_in"])
        if i >= 2:
            comp.wait_event(st["ev_out"])               # step i-2's outputs have left
        dt.dt_barrier(g, ALL, raw)
        dt.dt_reduce_scatter(g, ALL, st["in"], st["rs"], m, "bf16", "avg", raw)
        dt.dt_barrier(g, ALL, raw)
        dt.dt_all_gather(g, ALL, st["rs"], st["ag"], None, rows_ // P, cols * 2, 0, raw)
        st["ev_done"].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(st["ev_done"])
            for h, d in zip(st["h_out"], st["ag"]):
                h.copy_(d, non_blocking=True)
            st["ev_out"].record(s_out)

    for i in range(4):                                   # warm-up
        one(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    s_in.wait_stream(comp)
    s_out.wait_stream(comp)
    for i in range(steps):
        one(i)
    comp.wait_stream(s_out)
    t1.record(comp)
    torch.cuda.synchronize()
    rs_b, ag_b = step_bytes(P, rows_, cols)
    ms, value = aggregate(t0.elapsed_time(t1), (rs_b + ag_b) * steps, world, dev)
    h2d = sum(x.numel() * 2 for x in xs)
    d2h = sum(x.numel() * 2 for x in sets[0]["ag"])
    return ms, value, h2d, d2h


# Small invocations for ncu captures (the bench step itself serves its own
# ReduceScatter and AllGather): the kernel regex, the warm-up launches of that
# kernel to skip (-s) and what one case runs.  Sizes keep inputs larger than
# L2 where the workload has them and the device footprint to a few GB.
NCU_CASES = {
    "allreduce_small": ("reduce_vec_kernel", 2, "AllReduce kSum f32, P=2, 2^20 per rank"),
    "bucket": ("bucket_kernel", 14, "bucket AllReduce kAvg bf16, P=8, 200 tensors, 25 MiB buckets"),
    "all_to_all": ("copy_bulk_kernel", 2, "AllToAll bf16, P=8, [8192, 4096] per rank"),
    "all_to_all_p16": ("copy_bulk_kernel", 2, "AllToAll bf16, P=16, [8192, 2048] per rank"),
    "reduce_scatter_max_p16": ("reduce_vec_kernel", 2,
                               "ReduceScatter kMax bf16, P=16, 64 MiB per rank (sweep point)"),
    "uneven_all_gather": ("copy_bulk_kernel", 2,
                          "uneven AllGather int32, P=8, rows U[1, 2048] x 4096, per-rank outputs"),
    "barrier": ("barrier_kernel", 2, "signal-window barrier, P=16"),
    "allreduce_large": ("reduce_vec_kernel", 2, "AllReduce kSum f32, P=8, 64 MiB per rank"),
    "all_to_all_2d": ("copy2d_kernel", 2, "AllToAll S(0) -> S(1) bf16, P=8, [8192, 4096] per rank"),
    "small_gather": ("copy_vec_kernel", 2, "AllGather bf16, P=4, 256 KiB shards, per-rank outputs"),
    "reduce_scalar": ("reduce_scalar_kernel", 2,
                      "AllReduce kSum bf16, P=4, 16 MiB per rank, inputs and outputs at different offsets"),
    "reduce_shift": ("reduce_shift_kernel", 2,
                     "AllReduce kSum bf16, P=4, 16 MiB per rank, inputs at different offsets, aligned outputs"),
    "shift_gather": ("copy_shift_kernel", 2,
                     "AllGather bf16, P=4, 16 MiB shards 2 bytes past a boundary, aligned outputs"),
}


def run_ncu_case(name):
    """Two warm-up calls and three more of one collective, for an ncu capture
    (-k <regex> -s <skip> from NCU_CASES).  Prints one JSON line."""
    import torch
    from same_device_collective_gb300 import dt, workloads
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ALL = dt.DT_ALL_RANKS
    if name == "allreduce_small":
        xs = [x.to(dev) for x in workloads.allreduce_small().inputs]
        outs = [torch.empty_like(x) for x in xs]
        g = dt.dt_group_create(2, dev.index)
        call = lambda: dt.dt_allreduce(g, ALL, xs, outs, xs[0].numel(), "f32", "sum")
    elif name == "bucket":
        w = workloads.bucket_grads(device=str(dev))
        table = dt.pointer_table(w.inputs)
        cnt = np.asarray(w.meta["counts"], dtype=np.uint64)
        g = dt.dt_group_create(8, dev.index)
        call = lambda: dt.dt_bucket_allreduce(g, table, cnt, "bf16", "avg",
                                              workloads.BUCKET_CAP_BYTES)
    elif name == "all_to_all":
        w = workloads.all_to_all_tokens(rows=8192, device=str(dev))
        outs = [torch.empty_like(x) for x in w.inputs]
        nbytes = w.inputs[0].numel() * 2
        g = dt.dt_group_create(8, dev.index)
        call = lambda: dt.dt_all_to_all(g, ALL, w.inputs, outs, nbytes // 8)
    elif name == "all_to_all_p16":
        w = workloads.all_to_all_tokens(P=16, rows=8192, cols=2048, device=str(dev))
        outs = [torch.empty_like(x) for x in w.inputs]
        nbytes = w.inputs[0].numel() * 2
        g = dt.dt_group_create(16, dev.index)
        call = lambda: dt.dt_all_to_all(g, ALL, w.inputs, outs, nbytes // 16)
    elif name == "reduce_scatter_max_p16":
        w = workloads.sweep_inputs(4, 16, 64 << 20, "bf16", device=str(dev))
        n = w.inputs[0].numel()
        outs = [torch.empty(n // 16, dtype=torch.bfloat16, device=dev) for _ in range(16)]
        g = dt.dt_group_create(16, dev.index)
        call = lambda: dt.dt_reduce_scatter(g, ALL, w.inputs, outs, n // 16, "bf16", "max")
    elif name == "uneven_all_gather":
        w = workloads.uneven_gather(max_rows=2048, device=str(dev))
        rws = w.meta["rows"]
        outs = [torch.empty(sum(rws), 4096, dtype=torch.int32, device=dev) for _ in range(8)]
        g = dt.dt_group_create(8, dev.index)
        call = lambda: dt.dt_all_gather(g, ALL, w.inputs, outs, rws, 0, 4096 * 4)
    elif name == "barrier":
        g = dt.dt_group_create(16, dev.index)
        call = lambda: dt.dt_barrier(g)
    elif name == "allreduce_large":
        gen = torch.Generator(device=dev).manual_seed(4)
        n = 16 << 20
        xs = [torch.rand(n, generator=gen, device=dev) for _ in range(8)]
        outs = [torch.empty_like(x) for x in xs]
        g = dt.dt_group_create(8, dev.index)
        call = lambda: dt.dt_allreduce(g, ALL, xs, outs, n, "f32", "sum")
    elif name == "all_to_all_2d":
        w = workloads.all_to_all_tokens(rows=8192, device=str(dev))
        R8, C8 = w.inputs[0].shape
        outs = [torch.empty(8 * R8, C8 // 8, dtype=torch.bfloat16, device=dev) for _ in range(8)]
        g = dt.dt_group_create(8, dev.index)
        call = lambda: dt.dt_all_to_all_2d(g, ALL, w.inputs, outs, R8, C8, 2, 0, 1)
    elif name in ("small_gather", "shift_gather"):
        n = (128 << 10) if name == "small_gather" else (8 << 20)    # bf16 elements per shard
        off = 0 if name == "small_gather" else 1
        gen = torch.Generator(device=dev).manual_seed(4)
        base = [torch.rand(n + 8, generator=gen, device=dev).to(torch.bfloat16) for _ in range(4)]
        shards = [b_[off:off + n] for b_ in base]
        outs = [torch.empty(4 * n, dtype=torch.bfloat16, device=dev) for _ in range(4)]
        g = dt.dt_group_create(4, dev.index)
        call = lambda: dt.dt_all_gather(g, ALL, shards, outs, None, 1, n * 2)
    elif name in ("reduce_scalar", "reduce_shift"):
        n = 8 << 20
        gen = torch.Generator(device=dev).manual_seed(4)
        base = [torch.rand(n + 8, generator=gen, device=dev).to(torch.bfloat16) for _ in range(4)]
        xs = [b_[r:r + n] for r, b_ in enumerate(base)]          # offsets 0, 2, 4, 6 bytes
        if name == "reduce_shift":
            outs = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(4)]
        else:                                                   # outputs apart too
            obase = [torch.empty(n + 8, dtype=torch.bfloat16, device=dev) for _ in range(4)]
            outs = [b_[r:r + n] for r, b_ in enumerate(obase)]
        g = dt.dt_group_create(4, dev.index)
        call = lambda: dt.dt_allreduce(g, ALL, xs, outs, n, "bf16", "sum")
    else:
        raise ValueError(name)
    for _ in range(5):
        call()
    torch.cuda.synchronize()
    st = dt.dt_group_check(g)
    dt.dt_group_destroy(g)
    regex, skip, what = NCU_CASES[name]
    print(json.dumps({"ncu_case": name, "what": what, "calls": 5, "kernel_regex": regex,
                      "skip_launches": skip, "status_ok": st == dt.DT_OK}))
    return 0 if st == dt.DT_OK else 1


def summarize_timeline(rec, dt):
    """Per launch (grouped by grid id, in order of their first block's wait):
    kind, blocks, when work started and ended, and the gaps between launches;
    for a bucket kernel also its drain and ramp and its barrier block."""
    import numpy as np
    out = []
    grids = {}
    for r in rec:
        grids.setdefault(int(r["grid"]), []).append(r)
    launches = []
    for gid, rs in grids.items():
        rs = np.array(rs, dtype=rec.dtype)
        data = rs[rs["kind"] != 8]
        bar = rs[rs["kind"] == 8]
        if data.size == 0:
            continue
        ends = np.sort(data["t_end"].astype(np.int64))
        launches.append({
            "kind": dt.TIMELINE_KINDS.get(int(data["kind"][0]), str(int(data["kind"][0]))),
            "blocks": int(data.size),
            "work_start": int(data["t_waited"].min()), "work_end": int(ends[-1]),
            "first_end": int(ends[0]), "p90_end": int(ends[int(0.9 * (ends.size - 1))]),
            "barrier_end": int(bar["t_end"].max()) if bar.size else None})
    launches.sort(key=lambda x: x["work_start"])
    if not launches:
        return {"launches": 0}
    t0 = launches[0]["work_start"]
    prev = None
    for L in launches:
        e = {"kind": L["kind"], "blocks": L["blocks"],
             "start_us": round((L["work_start"] - t0) / 1e3, 3),
             "span_us": round((L["work_end"] - L["work_start"]) / 1e3, 3),
             "ramp_us": round((L["first_end"] - L["work_start"]) / 1e3, 3),
             "drain_us": round((L["work_end"] - L["p90_end"]) / 1e3, 3)}
        if L["barrier_end"] is not None:
            e["barrier_after_last_block_us"] = round((L["barrier_end"] - L["work_end"]) / 1e3, 3)
        if prev is not None:
            last = prev["barrier_end"] if prev["barrier_end"] is not None else prev["work_end"]
            e["gap_from_previous_us"] = round((L["work_start"] - last) / 1e3, 3)
        out.append(e)
        prev = L
    return {"launches": len(out), "per_launch": out}


def summarize_overlap(rec, dt):
    """Compute intervals from the marks around each GEMM (tags 2m, 2m + 1) and
    the collectives' launches: how much of the collectives' block time falls
    inside a GEMM interval."""
    import numpy as np
    marks = rec[rec["kind"] == 10]
    by_tag = {int(m["block"]): int(m["t_end"]) for m in marks}
    gemms = sorted((by_tag[2 * m], by_tag[2 * m + 1]) for m in range(len(by_tag) // 2)
                   if 2 * m in by_tag and 2 * m + 1 in by_tag)
    coll = rec[(rec["kind"] != 10) & (rec["kind"] != 8)]
    grids = {}
    for r in coll:
        grids.setdefault(int(r["grid"]), []).append(r)
    spans = sorted((int(np.min([x["t_waited"] for x in v])), int(np.max([x["t_end"] for x in v])))
                   for v in grids.values())

    def overlap(a, b):
        return max(0, min(a[1], b[1]) - max(a[0], b[0]))

    coll_ns = sum(e - s_ for s_, e in spans)
    inside = sum(overlap(sp, gm) for sp in spans for gm in gemms)
    t0 = min([g[0] for g in gemms] + [sp[0] for sp in spans]) if spans or gemms else 0
    t1 = max([g[1] for g in gemms] + [sp[1] for sp in spans]) if spans or gemms else 0
    gemm_ns = sum(e - s_ for s_, e in gemms)
    return {"gemms": len(gemms), "gemm_us": round(gemm_ns / 1e3, 1),
            "collective_launches": len(spans), "collective_us": round(coll_ns / 1e3, 1),
            "collective_us_inside_gemms": round(inside / 1e3, 1),
            "overlap_fraction_of_collective_time": round(inside / coll_ns, 3) if coll_ns else None,
            "first_to_last_us": round((t1 - t0) / 1e3, 1),
            "per_gemm_us": [round((e - s_) / 1e3, 1) for s_, e in gemms]}


def run_timeline(name):
    """A few calls of one workload on a library built with DT_TIMELINE=1, and
    the per-launch summary of their block timeline (one JSON line)."""
    import torch
    from same_device_collective_gb300 import dt, workloads
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ALL = dt.DT_ALL_RANKS
    try:
        dt.dt_timeline_start(1 << 20)
    except dt.DtError as ex:
        print(json.dumps({"timeline": name, "unavailable": f"{ex} (build with DT_TIMELINE=1)"}))
        return 1
    if name == "bucket":
        w = workloads.bucket_grads(device=str(dev))
        table = dt.pointer_table(w.inputs)
        cnt = np.asarray(w.meta["counts"], dtype=np.uint64)
        g = dt.dt_group_create(8, dev.index)
        call = lambda: dt.dt_bucket_allreduce(g, table, cnt, "bf16", "avg", workloads.BUCKET_CAP_BYTES)
        what = "bucket AllReduce kAvg bf16, P=8, 200 tensors, 25 MiB buckets: the third of 3 calls"
    elif name == "step":
        P, R, C = P_RANKS, ROWS, COLS
        w = workloads.rs_ag(seed=1, P=P, rows=R, cols=C, device=str(dev))
        rs = [torch.empty(R // P, C, dtype=torch.bfloat16, device=dev) for _ in range(P)]
        ag = [torch.empty(R, C, dtype=torch.bfloat16, device=dev) for _ in range(P)]
        g = dt.dt_group_create(P, dev.index)

        def call():
            dt.dt_barrier(g)
            dt.dt_reduce_scatter(g, ALL, w.inputs, rs, R // P * C, "bf16", "avg")
            dt.dt_barrier(g)
            dt.dt_all_gather(g, ALL, rs, ag, None, R // P, C * 2)
        what = "RS(avg)+AG step with barriers, P=4, bf16 [8192, 4096]: the third of 3 steps"
    elif name == "hsdp":
        h = HsdpSchedule(dt, dev)
        h.mark = lambda stream, tag: dt.dt_timeline_mark(stream, tag)
        call = h.pipelined
        what = ("pipelined post_backward schedule, 2 x 2 mesh, 8 modules, a bf16 GEMM standing in "
                "for each module's backward: the third of 3 runs")
        for _ in range(2):
            call()
        torch.cuda.synchronize()
        dt.dt_timeline_start(1 << 20)
        call()
        rec, n = dt.dt_timeline_read(1 << 20)
        ok = h.close()
        print(json.dumps({"timeline": name, "what": what, "records": n, "status_ok": ok,
                          **summarize_overlap(rec, dt)}))
        return 0 if ok else 1
    else:
        raise ValueError(name)
    for _ in range(2):
        call()
    torch.cuda.synchronize()
    dt.dt_timeline_start(1 << 20)
    torch.cuda._sleep(2_000_000)               # the host enqueues the call before it runs
    call()
    rec, n = dt.dt_timeline_read(1 << 20)
    ok = dt.dt_group_check(g) == dt.DT_OK
    dt.dt_group_destroy(g)
    print(json.dumps({"timeline": name, "what": what, "records": n, "status_ok": ok,
                      **summarize_timeline(rec, dt)}))
    return 0 if ok else 1


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from same_device_collective_gb300 import dt, workloads

    peak, peak_kind = measured_peak()
    P, rows_, cols = P_RANKS, ROWS, COLS
    w = workloads.rs_ag(seed=1, P=P, rows=rows_, cols=cols, device=str(dev))
    xs = w.inputs
    m = rows_ // P * cols
    rs = [torch.empty(rows_ // P, cols, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    ag = [torch.empty(rows_, cols, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    g = dt.dt_group_create(P, local)
    ALL = dt.DT_ALL_RANKS
    rs_b, ag_b = step_bytes()
    stream = torch.cuda.current_stream(dev)

    raw = stream.cuda_stream

    def step(ev=None):
        dt.dt_barrier(g, ALL, raw)
        if ev is not None:
            ev[0].record()
        dt.dt_reduce_scatter(g, ALL, xs, rs, m, "bf16", "avg", raw)
        if ev is not None:
            ev[1].record()
        dt.dt_barrier(g, ALL, raw)
        if ev is not None:
            ev[2].record()
        dt.dt_all_gather(g, ALL, rs, ag, None, rows_ // P, cols * 2, 0, raw)
        if ev is not None:
            ev[3].record()

    for _ in range(args.warmup):
        step()
    K = args.steps
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # timed region: K back-to-back steps, nothing between the launches, so the
    # kernels' programmatic dependent launches overlap each launch with the
    # previous kernel's tail.  A ~1 ms GPU sleep ahead of the start event (not
    # timed) lets the host enqueue the first steps before the event fires, so
    # the interval holds device time only, not the host's first calls.
    launches0 = dt.dt_launch_count()
    wall0 = time.time()
    torch.cuda._sleep(2_000_000)
    t_start.record()
    for _ in range(K):
        step()
    t_end.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    launches = dt.dt_launch_count() - launches0
    if world > 1:
        torch.distributed.barrier()
    time.sleep(0.2)
    clocks.stop()
    local_ms = t_start.elapsed_time(t_end)
    ms, value = aggregate(local_ms, (rs_b + ag_b) * K, world, dev)

    # per-kernel durations: a second pass with a CUDA event pair around each
    # ReduceScatter and AllGather launch; the events serialise the launches
    # (no overlap with the neighbouring kernels), so these are upper bounds
    K2 = min(K, 2000)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K2)]
    torch.cuda.synchronize()
    torch.cuda._sleep(2_000_000)          # as above: the host runs ahead of the GPU
    for i in range(K2):
        step(evs[i])
    torch.cuda.synchronize()
    rs_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / K2
    ag_ms = sum(e[2].elapsed_time(e[3]) for e in evs) / K2
    assert dt.dt_group_check(g) == dt.DT_OK

    if rs_ms >= ag_ms:
        dom, dom_bytes, dom_ms, key = "reduce_scatter (reduce_vec_kernel<bf16,avg,P<=4>)", rs_b, rs_ms, "reduce_scatter"
    else:
        dom, dom_bytes, dom_ms, key = "all_gather (copy_bulk_kernel, TMA)", ag_b, ag_ms, "all_gather"
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": ncu_traffic(key),
                "kernel": dom, "peak_kind": peak_kind,
                "algorithmic_bytes_per_launch": dom_bytes, "avg_launch_us": round(dom_ms * 1e3, 2),
                "timing": f"CUDA events around each launch over {K2} steps (serialised launches)",
                "per_kernel": {
                    "reduce_scatter": {"bytes": rs_b, "avg_us": round(rs_ms * 1e3, 2),
                                       "GB/s": round(rs_b / (rs_ms * 1e-3) / 1e9, 1)},
                    "all_gather": {"bytes": ag_b, "avg_us": round(ag_ms * 1e3, 2),
                                   "GB/s": round(ag_b / (ag_ms * 1e-3) / 1e9, 1)}}}

    # e2e: the same step through the public API with every step's four inputs
    # copied in from pinned host memory and its four gathered outputs copied
    # back, inside the timed region.  Steps are software-pipelined over two
    # device buffer sets: the inputs of step i+1 travel host->device and the
    # outputs of step i device->host (each on its own stream) while step i or
    # i+1 computes.
    e2e_steps = max(3, min(K, 50))
    e2e_ms, e2e_value, h2d, d2h = run_e2e(dt, g, xs, P, rows_, cols, m, e2e_steps, world, dev)

    rows_out = None
    if args.rows and world == 1:
        dt.dt_group_destroy(g)
        g = None
        rows_out = measure_rows(dt, dev, peak)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, el, reps = time_oracle(1024, min_seconds=10.0, max_reps=400)
        cpu = {"value": round(v, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"RS(avg)+AG on {P} ranks x bf16 [1024, {COLS}] (1/8 of the workload's "
                         f"rows, drawn with the same recipe), {reps} reps in {el:.1f} s, "
                         f"single-threaded C",
               "host": host_info(), "per_config": time_oracle_configs()}

    if g is not None:
        dt.dt_group_destroy(g)
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(ms / K, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "P": P, "rows": rows_, "cols": cols,
                       "op": "avg", "accumulate": "fp32",
                       "step": "barrier, reduce_scatter(avg), barrier, all_gather",
                       "bytes_per_step": rs_b + ag_b, "outputs": "per-rank",
                       "l2": "inputs larger than L2 (256 MiB of inputs per step vs 126.5 MB L2)",
                       "parallelism": f"replicas x{world}, P={P} logical ranks per GPU"},
            "frac_of_8TBs": round(value / world / NOMINAL_HBM_GBS, 4),
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "ms_per_step": round(e2e_ms / e2e_steps, 4),
                    "pipeline": "two buffer sets; H2D, step and D2H on three streams"},
            "gpu_launches": launches,
            "clocks": clocks.summary(wall0, wall1),
        }
        if rows_out is not None:
            line["rows"] = rows_out
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_sweep(args):
    """Every op at per-rank sizes 4 KiB .. 1 GiB (x4), P in {2, 4, 8, 16},
    fp32/bf16/int32, kSum/kMax: one JSON line per point on stdout.  Each point
    is a CUDA graph of back-to-back calls (no host gaps between launches),
    replayed and timed with CUDA events; points whose working set (inputs plus
    outputs) fits in L2 are marked "l2_resident"."""
    import torch
    from same_device_collective_gb300 import dt, workloads
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, _ = measured_peak()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    ALL = dt.DT_ALL_RANKS
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "i32": torch.int32}
    ranks = [int(x) for x in args.sweep_ranks.split(",")]
    sizes = [b for b in workloads.SWEEP_BYTES if b <= args.sweep_max_bytes]
    cap_stream = torch.cuda.Stream(dev)
    raw = cap_stream.cuda_stream

    def timed(fn, ws):
        calls = 100 if ws < (64 << 20) else (20 if ws < (4 << 30) else 5)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap_stream):
            fn()                                   # first call outside the capture
            with torch.cuda.graph(graph, stream=cap_stream):
                for _ in range(calls):
                    fn()
        graph.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(3):
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record()
            graph.replay()
            s1.record()
            s1.synchronize()
            ts.append(s0.elapsed_time(s1) / calls)
        del graph
        ts.sort()
        return ts[1]

    def emit(op, P, dtype, redop, nbytes, outputs, ms, alg_bytes, ws):
        gbs = alg_bytes / (ms * 1e-3) / 1e9
        print(json.dumps({"sweep": op, "P": P, "dtype": dtype, "op": redop,
                          "bytes_per_rank": nbytes, "outputs": outputs,
                          "us": round(ms * 1e3, 3), "GB/s": round(gbs, 1),
                          "frac_of_measured": round(gbs / peak, 4),
                          "frac_of_8TBs": round(gbs / NOMINAL_HBM_GBS, 4),
                          "l2_resident": ws <= l2}), flush=True)

    for P in ranks:
        g = dt.dt_group_create(P, 0)
        for nbytes in sizes:
            for dtype in ["f32", "bf16", "i32"]:
                w = workloads.sweep_inputs(4, P, nbytes, dtype, device=str(dev))
                xs = w.inputs
                n = xs[0].numel()
                es = 2 if dtype == "bf16" else 4
                free = torch.cuda.mem_get_info(dev)[0]
                per_rank = P * nbytes <= 0.6 * free
                outs = [torch.empty_like(x) for x in xs] if per_rank else [torch.empty_like(xs[0])] * P
                flags = 0 if per_rank else dt.DT_SHARED_OUTPUT
                m = n // P
                rs = [torch.empty(m, dtype=tdt[dtype], device=dev) for _ in range(P)]
                for redop in ["sum", "max"]:
                    ar_bytes = (2 * P if per_rank else P + 1) * n * es
                    ms = timed(lambda: dt.dt_allreduce(g, ALL, xs, outs, n, dtype, redop, flags, raw),
                               ar_bytes)
                    emit("allreduce", P, dtype, redop, nbytes, "per-rank" if per_rank else "shared",
                         ms, ar_bytes, ar_bytes)
                    rs_bytes = (P + 1) * n * es
                    ms = timed(lambda: dt.dt_reduce_scatter(g, ALL, xs, rs, m, dtype, redop, raw),
                               rs_bytes)
                    emit("reduce_scatter", P, dtype, redop, nbytes, "per-rank", ms, rs_bytes, rs_bytes)
                del outs, rs
                if dtype == "i32":
                    a2a = [torch.empty_like(x) for x in xs]
                    ms = timed(lambda: dt.dt_all_to_all(g, ALL, xs, a2a, nbytes // P, raw), 2 * P * nbytes)
                    emit("all_to_all", P, "bytes", None, nbytes, "per-rank", ms, 2 * P * nbytes,
                         2 * P * nbytes)
                    del a2a
                    free = torch.cuda.mem_get_info(dev)[0]
                    per_rank = P * P * nbytes <= 0.6 * free
                    if per_rank:
                        ag = [torch.empty(P * n, dtype=torch.int32, device=dev) for _ in range(P)]
                    else:
                        ag = [torch.empty(P * n, dtype=torch.int32, device=dev)] * P
                    ag_bytes = (P + P * P if per_rank else 2 * P) * nbytes
                    ms = timed(lambda: dt.dt_all_gather(g, ALL, xs, ag, None, 1, nbytes,
                                                        0 if per_rank else dt.DT_SHARED_OUTPUT, raw),
                               ag_bytes)
                    emit("all_gather", P, "bytes", None, nbytes, "per-rank" if per_rank else "shared",
                         ms, ag_bytes, ag_bytes)
                    del ag
                del w, xs
                torch.cuda.empty_cache()
        assert dt.dt_group_check(g) == dt.DT_OK
        dt.dt_group_destroy(g)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-rows", dest="rows", action="store_false")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="per-op size sweep (one JSON line per point) instead of the step")
    ap.add_argument("--sweep-ranks", default="2,4,8,16")
    ap.add_argument("--sweep-max-bytes", type=int, default=1 << 30)
    ap.add_argument("--row", choices=ROW_NAMES,
                    help="measure one collective at its own workload and print it")
    ap.add_argument("--ncu-case", choices=sorted(NCU_CASES),
                    help="run a few calls of one collective for an ncu capture (no timing)")
    ap.add_argument("--timeline", choices=["bucket", "step", "hsdp"],
                    help="per-block kernel timeline of one call (a DT_TIMELINE=1 build)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.ncu_case:
        return run_ncu_case(args.ncu_case)
    if args.timeline:
        return run_timeline(args.timeline)
    if args.row:
        import torch
        from same_device_collective_gb300 import dt
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps({"rows": measure_rows(dt, dev, measured_peak()[0], only=args.row)}))
        return 0
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
