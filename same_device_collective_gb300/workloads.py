"""Seeded synthetic workloads for the same-device collectives.

This module only draws random numbers and lays them out the way the pages'
workloads are shaped; it holds none of the collectives' arithmetic, so the
CUDA path and the CPU oracle can both read the bytes it produces.

Every generator is ``torch.Generator`` seeded per workload.  Small workloads
are drawn on the CPU (bit-identical on every host); the multi-GiB ones can be
drawn with a CUDA generator on the device and read back by whoever checks
them.  The recipe of each workload is in its docstring.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

GiB = 1 << 30
MiB = 1 << 20

# DDP's default gradient bucket: bucket_cap_mb = 25, read as 25 MiB.
BUCKET_CAP_BYTES = 25 * MiB

SWEEP_BYTES = [4096 * 4 ** k for k in range(10)]       # 4 KiB ... 1 GiB per rank
SWEEP_RANKS = [2, 4, 8, 16]


def _gen(seed: int, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def uniform_pm1(n: int, gen: torch.Generator, dtype=torch.float32, device="cpu") -> torch.Tensor:
    """n values uniform in [-1, 1), drawn in fp32 then cast."""
    x = torch.rand(n, generator=gen, device=device, dtype=torch.float32) * 2 - 1
    return x.to(dtype)


def normal(shape, gen: torch.Generator, std: float = 1.0, dtype=torch.bfloat16,
           device="cpu") -> torch.Tensor:
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(dtype)


@dataclass
class Workload:
    name: str
    P: int
    inputs: list                       # per-rank tensors
    meta: dict = field(default_factory=dict)


def allreduce_small(seed: int = 0, P: int = 2, n: int = 1 << 20) -> Workload:
    """AllReduce kSum: P ranks, each a contiguous fp32 tensor of n values
    uniform in [-1, 1), drawn rank 0 first from one CPU generator."""
    g = _gen(seed)
    xs = [uniform_pm1(n, g) for _ in range(P)]
    return Workload(f"allreduce_sum_f32_P{P}_n{n}", P, xs, {"n": n, "dtype": "f32", "op": "sum"})


def rs_ag(seed: int = 1, P: int = 4, rows: int = 8192, cols: int = 4096,
          device: str = "cpu") -> Workload:
    """ReduceScatter (AVG) then AllGatherIntoTensor: P ranks, each a bf16
    [rows, cols] tensor of N(0, 1) values (drawn in fp32, rounded to bf16),
    rank 0 first from one generator.  Shard r is rows [r*rows/P, (r+1)*rows/P)."""
    g = _gen(seed, device)
    xs = [normal((rows, cols), g, device=device) for _ in range(P)]
    return Workload(f"rs_avg_ag_bf16_P{P}_{rows}x{cols}", P, xs,
                    {"rows": rows, "cols": cols, "dtype": "bf16", "op": "avg"})


def bucket_counts(seed: int = 2, T: int = 200, lo: float = 1e3, hi: float = 4e6) -> list:
    """T element counts log-uniform in [lo, hi]: floor(exp(ln lo + u (ln hi - ln lo)))
    with u uniform in [0, 1) drawn in fp64 from a CPU generator."""
    g = _gen(seed)
    u = torch.rand(T, generator=g, dtype=torch.float64)
    a, b = math.log(lo), math.log(hi)
    return [int(math.floor(math.exp(a + float(ui) * (b - a)))) for ui in u]


def bucket_grads(seed: int = 2, P: int = 8, T: int = 200, lo: float = 1e3, hi: float = 4e6,
                 std: float = 1e-3, dtype=torch.bfloat16, device: str = "cpu",
                 counts: list | None = None) -> Workload:
    """Fused gradient-bucket all-reduce: T gradient tensors per rank, counts
    from ``bucket_counts`` (same shapes on every rank), values N(0, std) drawn
    tensor by tensor, rank 0 first within a tensor, then rounded to dtype.
    inputs[t][p] is rank p's gradient t."""
    if counts is None:
        counts = bucket_counts(seed, T, lo, hi)
    g = _gen(seed + 1000, device)
    grads = [[normal(c, g, std=std, dtype=dtype, device=device) for _ in range(P)]
             for c in counts]
    return Workload(f"bucket_avg_{'bf16' if dtype == torch.bfloat16 else 'f32'}_P{P}_T{len(counts)}",
                    P, grads, {"counts": counts, "cap_bytes": BUCKET_CAP_BYTES})


def all_to_all_tokens(seed: int = 3, P: int = 8, rows: int = 65536, cols: int = 4096,
                      device: str = "cpu") -> Workload:
    """AllToAll: P ranks, each a bf16 [rows, cols] token matrix of N(0, 1)
    values, split along dim 0 into P equal chunks; chunk j goes to rank j."""
    g = _gen(seed, device)
    xs = [normal((rows, cols), g, device=device) for _ in range(P)]
    return Workload(f"all_to_all_bf16_P{P}_{rows}x{cols}", P, xs, {"rows": rows, "cols": cols})


def uneven_rows(seed: int = 3, P: int = 8, max_rows: int = 16384) -> list:
    """Per-rank row counts uniform in [1, max_rows] from a CPU generator."""
    g = _gen(seed + 2000)
    return [int(v) for v in torch.randint(1, max_rows + 1, (P,), generator=g)]


def uneven_gather(seed: int = 3, P: int = 8, max_rows: int = 16384, cols: int = 4096,
                  device: str = "cpu", rows: list | None = None) -> Workload:
    """Uneven-shard AllGather: rank r holds rows[r] rows (``uneven_rows``) of
    `cols` int32 values uniform over [-2^31, 2^31 - 2]."""
    if rows is None:
        rows = uneven_rows(seed, P, max_rows)
    g = _gen(seed + 3000, device)
    xs = [torch.randint(-2 ** 31, 2 ** 31 - 1, (c, cols), generator=g, device=device,
                        dtype=torch.int32) for c in rows]
    return Workload(f"uneven_all_gather_i32_P{P}_{cols}cols", P, xs, {"rows": rows, "cols": cols})


def sweep_inputs(seed: int, P: int, nbytes: int, dtype: str, device: str = "cpu") -> Workload:
    """Sweep point: P ranks of nbytes each; fp32 / bf16 uniform in [-1, 1),
    int32 uniform in [-2^20, 2^20]."""
    g = _gen(seed, device)
    es = 2 if dtype == "bf16" else 4
    n = nbytes // es
    if dtype == "i32":
        xs = [torch.randint(-2 ** 20, 2 ** 20 + 1, (n,), generator=g, device=device,
                            dtype=torch.int32) for _ in range(P)]
    else:
        td = torch.bfloat16 if dtype == "bf16" else torch.float32
        xs = [uniform_pm1(n, g, td, device) for _ in range(P)]
    return Workload(f"sweep_{dtype}_P{P}_{nbytes}B", P, xs, {"n": n, "dtype": dtype})
