"""Seeded random collective calls against the oracle.

Each case draws a rank count, sizes, dtype, op, byte offsets (16-byte aligned
or not) and output mode, so that calls land on every launch shape the library
picks between: element-wise and vector reductions, the small register copy,
and the bulk copy's gather, split and AllToAll shapes, including sizes at
their thresholds (16 MiB of source, 4 and 16 tiles per SM).  Every output is
compared with the oracle bit for bit and every output sits between guard
bytes that must survive.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import ELEM, TORCH_DTYPE, bytes_of, group, host

pytestmark = pytest.mark.gpu

GUARD = 4096


@pytest.fixture(scope="module")
def dt():
    from same_device_collective_gb300 import dt as mod
    assert torch.cuda.is_available()
    return mod


def boxed(nbytes: int, shift: int, gen: torch.Generator, fill=None):
    """A uint8 view of nbytes at byte offset GUARD + shift inside a larger
    buffer whose other bytes hold 0x5A; returns (base, view)."""
    base = torch.full((GUARD + shift + nbytes + GUARD,), 0x5A, dtype=torch.uint8, device="cuda")
    v = base[GUARD + shift:GUARD + shift + nbytes]
    if fill is not None:
        v.copy_(fill)
    else:
        v.copy_(torch.randint(0, 256, (nbytes,), generator=gen, dtype=torch.uint8, device="cuda"))
    return base, v


def guards_ok(base: torch.Tensor, shift: int, nbytes: int) -> bool:
    lo, hi = GUARD + shift, GUARD + shift + nbytes
    return bool((base[:lo] == 0x5A).all()) and bool((base[hi:] == 0x5A).all())


def finite_values(nbytes, dtype, gen):
    n = nbytes // ELEM[dtype]
    if dtype == "i32":
        x = torch.randint(-2 ** 20, 2 ** 20, (n,), generator=gen, device="cuda", dtype=torch.int32)
    else:
        x = (torch.rand(n, generator=gen, device="cuda") * 2 - 1).to(TORCH_DTYPE[dtype])
    return x.view(torch.uint8)


@pytest.mark.parametrize("case", range(24))
def test_random_reductions(dt, case):
    rng = np.random.default_rng(1000 + case)
    P = int(rng.integers(1, 17))
    dtype, op = [("f32", "sum"), ("f32", "avg"), ("f32", "max"), ("bf16", "sum"), ("bf16", "avg"),
                 ("bf16", "min"), ("i32", "sum"), ("i32", "max"), ("bf16", "sum_stepwise")][
        int(rng.integers(0, 9))]
    es = ELEM[dtype]
    m = int(rng.choice([1, 7, 255, 4097, 65_536 + 3, int(rng.integers(1, 300_000))]))
    shift = int(rng.choice([0, 0, es, 4 * es]))                 # mostly aligned
    gen = torch.Generator(device="cuda").manual_seed(case)
    ins = [boxed(P * m * es, shift, gen, finite_values(P * m * es, dtype, gen)) for _ in range(P)]
    xs = [v.view(TORCH_DTYPE[dtype]) for _, v in ins]
    ar = [boxed(P * m * es, shift, gen) for _ in range(P)]
    rs = [boxed(m * es, shift, gen) for _ in range(P)]
    with group(P) as g:
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, [v.view(TORCH_DTYPE[dtype]) for _, v in ar],
                        P * m, dtype, op)
        dt.dt_reduce_scatter(g, dt.DT_ALL_RANKS, xs, [v.view(TORCH_DTYPE[dtype]) for _, v in rs],
                             m, dtype, op)
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
    hx = [host(x) for x in xs]
    want = oracle.allreduce(dtype, op, hx)
    for q, (b, v) in enumerate(ar):
        assert guards_ok(b, shift, P * m * es), f"allreduce guard rank {q}"
        assert np.array_equal(bytes_of(host(v)), bytes_of(want[q])), f"allreduce rank {q}"
    want = oracle.reduce_scatter(dtype, op, hx)
    for r, (b, v) in enumerate(rs):
        assert guards_ok(b, shift, m * es), f"reduce_scatter guard rank {r}"
        assert np.array_equal(bytes_of(host(v)), bytes_of(want[r])), f"reduce_scatter rank {r}"


@pytest.mark.parametrize("case", range(24))
def test_random_copies(dt, case):
    rng = np.random.default_rng(2000 + case)
    P = int(rng.integers(1, 17))
    shift = int(rng.choice([0, 0, 0, 4]))
    gen = torch.Generator(device="cuda").manual_seed(100 + case)
    # AllToAll chunk sizes around the copy thresholds (16-byte multiples when aligned)
    chunk = int(rng.choice([16, 4096, 48 * 1024, (16 << 20) // max(P * P, 1), 1 << 20,
                            (3 << 20) // max(P, 1)]))
    chunk = max(16, chunk // 16 * 16) + (0 if shift == 0 else 12)
    xs = [boxed(P * chunk, shift, gen) for _ in range(P)]
    outs = [boxed(P * chunk, shift, gen) for _ in range(P)]
    # uneven AllGather, per-rank or shared output
    row_bytes = int(rng.choice([16, 4096, 16384])) + (0 if shift == 0 else 4)
    rows = [int(v) for v in rng.integers(0, int(rng.choice([4, 300, 2000])), P)]
    rows[int(rng.integers(0, P))] += 1                         # at least one row
    total = sum(rows) * row_bytes
    shared = bool(rng.integers(0, 2)) or P * total > (1 << 30)   # bound host memory
    shards = [boxed(c * row_bytes, shift, gen) for c in rows]
    gath = [boxed(total, shift, gen)] if shared else [boxed(total, shift, gen) for _ in range(P)]
    with group(P) as g:
        dt.dt_all_to_all(g, dt.DT_ALL_RANKS, [v for _, v in xs], [v for _, v in outs], chunk)
        dt.dt_all_gather(g, dt.DT_ALL_RANKS, [v for _, v in shards],
                         [gath[0][1]] * P if shared else [v for _, v in gath], rows, 0, row_bytes,
                         dt.DT_SHARED_OUTPUT if shared else 0)
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
    want = oracle.all_to_all([host(v) for _, v in xs])
    for j, (b, v) in enumerate(outs):
        assert guards_ok(b, shift, P * chunk), f"all_to_all guard rank {j}"
        assert np.array_equal(host(v), want[j]), f"all_to_all rank {j} (P={P}, chunk={chunk})"
    want = oracle.all_gather([host(v) for _, v in shards], rows, row_bytes)
    for q, (b, v) in enumerate(gath):
        assert guards_ok(b, shift, total), f"all_gather guard output {q}"
        assert np.array_equal(host(v), want[q]), f"all_gather output {q} (P={P}, rows={rows})"
