"""No collective writes outside its outputs.

Every output buffer (and every buffer a call updates in place) sits inside a
larger allocation whose first and last 64 KiB hold a known byte pattern; after
each call both guard zones must still hold it, every input must be unchanged
and the result must equal the oracle's.  Sizes are ragged on purpose: vector
tails, partial bulk-copy tiles (16 and 32 KiB), zero-row ranks, buffers that
start 4 bytes off a 16-byte boundary, and empty tensors in a bucket.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import ELEM, TORCH_DTYPE, bytes_of, group, host, rand_inputs

pytestmark = pytest.mark.gpu

GUARD = 64 << 10
PATTERN = 0xA5


@pytest.fixture(scope="module")
def dt():
    from same_device_collective_gb300 import dt as mod
    assert torch.cuda.is_available()
    return mod


class Guarded:
    """nbytes of payload at byte offset GUARD + shift of a pattern-filled allocation."""

    def __init__(self, nbytes: int, shift: int = 0):
        self.base = torch.full((GUARD + shift + nbytes + GUARD,), PATTERN, dtype=torch.uint8,
                               device="cuda")
        self.lo, self.hi = GUARD + shift, GUARD + shift + nbytes

    def view(self, dtype: torch.dtype) -> torch.Tensor:
        return self.base[self.lo:self.hi].view(dtype)

    def intact(self) -> bool:
        return bool((self.base[:self.lo] == PATTERN).all()) and bool((self.base[self.hi:] == PATTERN).all())


def guarded_like(n: int, dtype: str, shift: int = 0, fill: torch.Tensor | None = None):
    g = Guarded(n * ELEM[dtype], shift)
    v = g.view(TORCH_DTYPE[dtype])
    if fill is not None:
        v.copy_(fill)
    return g, v


def assert_same(got, want, what):
    g, w = bytes_of(got), bytes_of(want)
    assert g.size == w.size and np.array_equal(g, w), what


def snapshot(ts):
    return [host(t).copy() for t in ts]


def unchanged(ts, snap):
    return all(np.array_equal(bytes_of(host(t)), bytes_of(s)) for t, s in zip(ts, snap))


# --------------------------------------------------------------- AllReduce
@pytest.mark.parametrize("dtype,op", [("f32", "sum"), ("bf16", "avg"), ("i32", "max")])
@pytest.mark.parametrize("n", [1, 7, 4095, 100_003])
@pytest.mark.parametrize("shift", [0, 4])
def test_allreduce_writes_only_its_outputs(dt, dtype, op, n, shift):
    P = 3
    xs = rand_inputs(P, n, dtype, n % 97)
    snap = snapshot(xs)
    want = oracle.allreduce(dtype, op, snap)
    outs = [guarded_like(n, dtype, shift) for _ in range(P)]
    shared = guarded_like(n, dtype, shift)
    inplace = [guarded_like(n, dtype, shift, fill=x) for x in xs]
    with group(P) as g:
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, [v for _, v in outs], n, dtype, op)
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, [shared[1]] * P, n, dtype, op,
                        flags=dt.DT_SHARED_OUTPUT)
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, [v for _, v in inplace], [v for _, v in inplace], n,
                        dtype, op)
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
    assert unchanged(xs, snap)
    for q in range(P):
        assert outs[q][0].intact() and inplace[q][0].intact(), f"rank {q}"
        assert_same(host(outs[q][1]), want[q], f"per-rank rank {q}")
        assert_same(host(inplace[q][1]), want[q], f"in place rank {q}")
    assert shared[0].intact()
    assert_same(host(shared[1]), want[0], "shared")


# ----------------------------------------------------------- ReduceScatter
@pytest.mark.parametrize("dtype,op", [("bf16", "avg"), ("f32", "min")])
@pytest.mark.parametrize("m", [1, 5, 4099, 40_000])
@pytest.mark.parametrize("shift", [0, 4])
def test_reduce_scatter_writes_only_its_outputs(dt, dtype, op, m, shift):
    P = 3
    xs = rand_inputs(P, P * m, dtype, m % 89)
    snap = snapshot(xs)
    want = oracle.reduce_scatter(dtype, op, snap)
    outs = [guarded_like(m, dtype, shift) for _ in range(P)]
    with group(P) as g:
        dt.dt_reduce_scatter(g, dt.DT_ALL_RANKS, xs, [v for _, v in outs], m, dtype, op)
        torch.cuda.synchronize()
    assert unchanged(xs, snap)
    for r in range(P):
        assert outs[r][0].intact(), f"rank {r}"
        assert_same(host(outs[r][1]), want[r], f"rank {r}")


# --------------------------------------------------------------- AllGather
@pytest.mark.parametrize("rows,row_bytes", [([2, 2, 2], 12), ([0, 5, 9], 16), ([3, 7, 2], 16384),
                                            ([1, 0, 40], 4096)])
@pytest.mark.parametrize("shift", [0, 4])
def test_all_gather_writes_only_its_outputs(dt, rows, row_bytes, shift):
    P = 3
    gen = torch.Generator().manual_seed(sum(rows) + row_bytes)
    xs = [torch.randint(0, 256, (c * row_bytes,), generator=gen, dtype=torch.uint8).cuda()
          for c in rows]
    snap = snapshot(xs)
    total = sum(rows) * row_bytes
    want = oracle.all_gather_one(snap, rows, row_bytes)
    outs = [Guarded(total, shift) for _ in range(P)]
    shared = Guarded(total, shift)
    with group(P) as g:
        dt.dt_all_gather(g, dt.DT_ALL_RANKS, xs, [o.view(torch.uint8) for o in outs], rows, 0,
                         row_bytes)
        dt.dt_all_gather(g, dt.DT_ALL_RANKS, xs, [shared.view(torch.uint8)] * P, rows, 0,
                         row_bytes, flags=dt.DT_SHARED_OUTPUT)
        torch.cuda.synchronize()
    assert unchanged(xs, snap)
    for q, o in enumerate(outs + [shared]):
        assert o.intact(), f"output {q}"
        assert_same(host(o.view(torch.uint8)), want, f"output {q}")


# ---------------------------------------------------------------- AllToAll
@pytest.mark.parametrize("P", [3, 8])
@pytest.mark.parametrize("chunk_bytes", [12, 16, 48, 40_000])
def test_all_to_all_writes_only_its_outputs(dt, P, chunk_bytes):
    gen = torch.Generator().manual_seed(P * chunk_bytes)
    xs = [torch.randint(0, 256, (P * chunk_bytes,), generator=gen, dtype=torch.uint8).cuda()
          for _ in range(P)]
    snap = snapshot(xs)
    want = oracle.all_to_all(snap)
    outs = [Guarded(P * chunk_bytes) for _ in range(P)]
    with group(P) as g:
        dt.dt_all_to_all(g, dt.DT_ALL_RANKS, xs, [o.view(torch.uint8) for o in outs], chunk_bytes)
        torch.cuda.synchronize()
    assert unchanged(xs, snap)
    for j, o in enumerate(outs):
        assert o.intact(), f"rank {j}"
        assert_same(host(o.view(torch.uint8)), want[j], f"rank {j}")


@pytest.mark.parametrize("P,chunk_bytes", [(16, 7 * 16384 + 48), (8, (2 << 20) + 48),
                                           (4, (1 << 20) + 48)])
def test_bulk_all_to_all_shapes_write_only_their_outputs(dt, P, chunk_bytes):
    # The bulk-copy shapes of an AllToAll, each segment ending in a 48-byte
    # partial tile: 16 ranks of ~1.8 MiB (data fits in L2: four stages, three
    # blocks per SM), 8 ranks of ~16 MiB (data larger than half of L2: twelve
    # stages, one block per SM) and 4 ranks of ~4 MiB (16 segments: 16 KiB x
    # 4 stages, three blocks per SM).
    gen = torch.Generator(device="cuda").manual_seed(P + chunk_bytes)
    xs = [torch.randint(0, 256, (P * chunk_bytes,), generator=gen, dtype=torch.uint8, device="cuda")
          for _ in range(P)]
    snap = snapshot(xs)
    want = oracle.all_to_all(snap)
    outs = [Guarded(P * chunk_bytes) for _ in range(P)]
    with group(P) as g:
        dt.dt_all_to_all(g, dt.DT_ALL_RANKS, xs, [o.view(torch.uint8) for o in outs], chunk_bytes)
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
    assert unchanged(xs, snap)
    for j, o in enumerate(outs):
        assert o.intact(), f"rank {j}"
        assert_same(host(o.view(torch.uint8)), want[j], f"rank {j}")


# ------------------------------------------------------- bucket all-reduce
@pytest.mark.parametrize("dtype,op", [("bf16", "avg"), ("f32", "sum")])
@pytest.mark.parametrize("cap", [4096, 25 << 20])
@pytest.mark.parametrize("shift", [0, 4])
@pytest.mark.parametrize("static", [False, True])
def test_bucket_allreduce_writes_only_its_gradients(dt, dtype, op, cap, shift, static):
    P = 3
    counts = [1, 7, 4095, 70_001, 0, 33]
    gen = torch.Generator().manual_seed(cap % 1000 + shift)
    grads = []
    for c in counts:
        row = []
        for _ in range(P):
            x = (torch.randn(c, generator=gen) * 1e-3).to(TORCH_DTYPE[dtype])
            row.append(guarded_like(c, dtype, shift, fill=x.cuda()))
        grads.append(row)
    ref = [[host(v).copy() for _, v in row] for row in grads]
    views = [[v for _, v in row] for row in grads]
    if static:
        dt.dt_bucket_allreduce_static(P, views, counts, dtype, op, bucket_cap_bytes=cap)
        torch.cuda.synchronize()
    else:
        with group(P) as g:
            dt.dt_bucket_allreduce(g, views, counts, dtype, op, bucket_cap_bytes=cap)
            torch.cuda.synchronize()
            assert dt.dt_group_check(g) == dt.DT_OK
    oracle.bucket_allreduce(dtype, op, ref)
    for t in range(len(counts)):
        for p in range(P):
            assert grads[t][p][0].intact(), f"tensor {t} rank {p}"
            assert_same(host(views[t][p]), ref[t][p], f"tensor {t} rank {p}")


# -------------------------------------------------------------- placements
def test_placement_conversions_write_only_their_outputs(dt):
    P, R, C = 3, 6, 10                          # int32 [6, 10] per rank: 40-byte rows
    gen = torch.Generator().manual_seed(7)
    full = [torch.randint(-1000, 1000, (R, C), generator=gen, dtype=torch.int32).cuda()
            for _ in range(P)]
    snap = snapshot(full)
    shards = [Guarded(R // P * C * 4) for _ in range(P)]
    vec = [Guarded(R // P * C * 4) for _ in range(P * P)]
    a2a = [Guarded(R * C * 4) for _ in range(P)]            # S(1) -> S(0): [R / P, P * C]
    with group(P) as g:
        dt.dt_replicate_to_shard(g, dt.DT_ALL_RANKS, full, [s.view(torch.int32) for s in shards],
                                 None, R, C * 4)
        torch.cuda.synchronize()
        shard_in = [s.view(torch.int32) for s in shards]
        shard_snap = snapshot(shard_in)
        dt.dt_all_gather_into_vec(g, dt.DT_ALL_RANKS, shard_in, [v.view(torch.int32) for v in vec],
                                  None, R // P, C * 4)
        dt.dt_all_to_all_2d(g, dt.DT_ALL_RANKS, full, [o.view(torch.int32) for o in a2a],
                            R, C, 4, 1, 0)
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
    assert unchanged(full, snap) and unchanged(shard_in, shard_snap)
    want = oracle.replicate_to_shard(snap, R, C * 4)
    for r, sh in enumerate(shards):
        assert sh.intact(), f"shard {r}"
        assert_same(shard_snap[r], want[r], f"shard {r}")
    want_vec = oracle.all_gather_into_vec(shard_snap, [R // P] * P, C * 4)
    for i, v in enumerate(vec):
        assert v.intact(), f"vector slot {i}"
        assert_same(host(v.view(torch.int32)), want_vec[i], f"vector slot {i}")
    want_a2a = oracle.all_to_all_2d([x.reshape(R, C) for x in snap], 1, 0)
    for j, o in enumerate(a2a):
        assert o.intact(), f"all-to-all rank {j}"
        assert_same(host(o.view(torch.int32)), want_a2a[j], f"all-to-all rank {j}")


@pytest.mark.parametrize("rows,shared", [([8193, 8190], False), ([3073, 3070], True),
                                         ([1025, 1023, 1024, 1021], False)])
def test_large_gathers_in_waves_write_only_their_outputs(dt, rows, shared):
    # Big enough for the bulk copy's multi-wave grids: per-rank outputs of two
    # ~128 MiB shards take 96 KiB tiles in 8 waves, a shared output of two
    # ~48 MiB shards 32 KiB tiles in 8 waves, per-rank outputs of four ~16 MiB
    # shards 32 KiB tiles on two blocks per SM in 4 waves; every shard ends in
    # a partial tile.
    P, row_bytes = len(rows), 16384
    gen = torch.Generator(device="cuda").manual_seed(sum(rows))
    xs = [torch.randint(0, 256, (c * row_bytes,), generator=gen, device="cuda", dtype=torch.uint8)
          for c in rows]
    total = sum(rows) * row_bytes
    # 16-byte-aligned outputs: the bulk-copy path (a misaligned one takes the byte kernel)
    outs = [Guarded(total)] if shared else [Guarded(total) for _ in range(P)]
    with group(P) as g:
        dt.dt_all_gather(g, dt.DT_ALL_RANKS, xs, [o.view(torch.uint8) for o in outs] * (P if shared else 1),
                         rows, 0, row_bytes, flags=dt.DT_SHARED_OUTPUT if shared else 0)
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
    want = torch.cat(xs)
    for q, o in enumerate(outs):
        assert o.intact(), f"output {q}"
        assert torch.equal(o.view(torch.uint8), want), f"output {q}"
