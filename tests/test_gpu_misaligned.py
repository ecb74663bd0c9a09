"""Buffers that do not start on a 16-byte boundary, bit-exact against the oracle.

Two layouts reach different kernels:
- every buffer of a call (or of a ReduceScatter shard) lies the same distance
  past a 16-byte boundary -- views of the same offset into larger tensors.
  The reductions run their vector kernel from each buffer's first boundary
  and take the elements before it on the element path; the copies run their
  vector or bulk-copy kernels on the aligned middle of every segment and copy
  the edge bytes alongside;
- sources and destinations at different offsets (or rows of a byte count
  that is not a multiple of 16): the copies align every store and shift the
  source into place (a funnel shift across two aligned source vectors); the
  reductions do the same for inputs at their own offsets when the outputs
  share one, and otherwise reduce element by element.
Every output sits between two guard zones of a known byte pattern, which must
survive the call; inputs must be unchanged.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import ELEM, TORCH_DTYPE, bytes_of, group, host, rand_inputs

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0x5A


@pytest.fixture(scope="module")
def dt():
    from same_device_collective_gb300 import dt as mod
    assert torch.cuda.is_available()
    return mod


class Guarded:
    """nbytes at byte offset GUARD + shift of a pattern-filled allocation
    (the allocation itself starts on a 512-byte boundary)."""

    def __init__(self, nbytes: int, shift: int = 0):
        self.base = torch.full((GUARD + shift + nbytes + GUARD,), PATTERN, dtype=torch.uint8,
                               device="cuda")
        self.lo, self.hi = GUARD + shift, GUARD + shift + nbytes

    def view(self, dtype) -> torch.Tensor:
        return self.base[self.lo:self.hi].view(dtype)

    def intact(self) -> bool:
        return bool((self.base[:self.lo] == PATTERN).all()) and bool((self.base[self.hi:] == PATTERN).all())


def placed(x: torch.Tensor, shift: int):
    """A copy of x at byte offset `shift` past a 16-byte boundary."""
    g = Guarded(x.numel() * x.element_size(), shift)
    v = g.view(x.dtype)
    v.copy_(x.reshape(-1))
    return g, v


def empty_at(nbytes: int, dtype, shift: int):
    g = Guarded(nbytes, shift)
    return g, g.view(dtype)


def assert_same(got, want, what):
    g, w = bytes_of(got), bytes_of(want)
    assert g.size == w.size, what
    if not np.array_equal(g, w):
        bad = np.nonzero(g != w)[0]
        raise AssertionError(f"{what}: {bad.size} bytes differ, first at byte {bad[0]}")


# ------------------------------------------------------------- reductions
@pytest.mark.parametrize("dtype,op", [("bf16", "avg"), ("bf16", "sum_stepwise"), ("f32", "sum"),
                                      ("f32", "max"), ("i32", "sum"), ("bf16", "min")])
@pytest.mark.parametrize("elems_off", [1, 3, 7])
@pytest.mark.parametrize("n", [1, 5, 4099, 100_003])
def test_allreduce_shared_offset(dt, dtype, op, elems_off, n):
    P = 4
    shift = elems_off * ELEM[dtype] % 16
    xs = rand_inputs(P, n, dtype, 7 * n + elems_off)
    snap = [host(x).copy() for x in xs]
    want = oracle.allreduce(dtype, op, snap)
    ins = [placed(x, shift) for x in xs]
    outs = [empty_at(n * ELEM[dtype], TORCH_DTYPE[dtype], shift) for _ in range(P)]
    with group(P) as g:
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, [v for _, v in ins], [v for _, v in outs], n, dtype, op)
        torch.cuda.synchronize()
    for q, (gd, v) in enumerate(outs):
        assert_same(host(v), want[q], f"rank {q}")
        assert gd.intact(), f"guard of rank {q}"
    for (gd, v), s in zip(ins, snap):
        assert np.array_equal(bytes_of(host(v)), bytes_of(s)) and gd.intact()


@pytest.mark.parametrize("dtype,op", [("bf16", "avg"), ("bf16", "sum_stepwise"), ("f32", "sum"),
                                      ("f32", "min"), ("i32", "sum"), ("bf16", "max")])
@pytest.mark.parametrize("P", [2, 3, 8, 16])
@pytest.mark.parametrize("n", [1, 9, 4099, 100_003])
@pytest.mark.parametrize("out_layout", ["shared", "apart"])
def test_allreduce_inputs_at_their_own_offsets(dt, dtype, op, P, n, out_layout):
    # input r starts (3 r) mod 8 elements past a 16-byte boundary; with the
    # outputs at one offset the inputs are read as aligned vectors and
    # shifted into place, with outputs apart the call takes the element path
    es = ELEM[dtype]
    xs = rand_inputs(P, n, dtype, 3 * n + P)
    snap = [host(x).copy() for x in xs]
    want = oracle.allreduce(dtype, op, snap)
    ins = [placed(x, (3 * r * es) % 16) for r, x in enumerate(xs)]
    outs = [empty_at(n * es, TORCH_DTYPE[dtype], (es if out_layout == "shared" else q * es) % 16)
            for q in range(P)]
    with group(P) as g:
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, [v for _, v in ins], [v for _, v in outs], n, dtype, op)
        torch.cuda.synchronize()
    for q, (gd, v) in enumerate(outs):
        assert_same(host(v), want[q], f"rank {q}")
        assert gd.intact(), f"guard of rank {q}"


@pytest.mark.parametrize("dtype,op", [("bf16", "avg"), ("f32", "max"), ("i32", "sum")])
@pytest.mark.parametrize("P", [2, 5, 16])
@pytest.mark.parametrize("m", [1, 31, 4093, 20_001])
def test_reduce_scatter_inputs_at_their_own_offsets(dt, dtype, op, P, m):
    es = ELEM[dtype]
    xs = rand_inputs(P, P * m, dtype, 5 * m + P)
    want = oracle.reduce_scatter(dtype, op, [host(x) for x in xs])
    ins = [placed(x, (5 * r * es) % 16) for r, x in enumerate(xs)]
    outs = [empty_at(m * es, TORCH_DTYPE[dtype], (j * es) % 16) for j in range(P)]
    with group(P) as g:
        dt.dt_reduce_scatter(g, dt.DT_ALL_RANKS, [v for _, v in ins], [v for _, v in outs], m, dtype, op)
        torch.cuda.synchronize()
    for j, (gd, v) in enumerate(outs):
        assert_same(host(v), want[j], f"shard {j}")
        assert gd.intact(), f"guard of shard {j}"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_allreduce_shared_offset_in_place(dt, dtype):
    P, n = 3, 65_537
    shift = 2 * ELEM[dtype] % 16
    xs = rand_inputs(P, n, dtype, 5)
    want = oracle.allreduce(dtype, "sum", [host(x) for x in xs])
    bufs = [placed(x, shift) for x in xs]
    with group(P) as g:
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, [v for _, v in bufs], [v for _, v in bufs], n, dtype, "sum")
        torch.cuda.synchronize()
    for q, (gd, v) in enumerate(bufs):
        assert_same(host(v), want[q], f"rank {q}")
        assert gd.intact()


@pytest.mark.parametrize("dtype,op", [("bf16", "avg"), ("f32", "sum"), ("i32", "max")])
@pytest.mark.parametrize("m", [4096, 4093, 1, 77])
@pytest.mark.parametrize("elems_off", [0, 1, 5])
@pytest.mark.parametrize("P", [2, 3, 8])
def test_reduce_scatter_shard_offsets(dt, dtype, op, m, elems_off, P):
    # inputs share an offset; out[j] sits where shard j of the inputs sits
    # relative to a 16-byte boundary.  Shards of whole 16-byte vectors then
    # take the vector kernel from the first boundary; the others (m odd: the
    # shards' offsets differ) the element path.
    es = ELEM[dtype]
    xs = rand_inputs(P, P * m, dtype, 31 * m + P)
    snap = [host(x).copy() for x in xs]
    want = oracle.reduce_scatter(dtype, op, snap)
    shift = elems_off * es % 16
    ins = [placed(x, shift) for x in xs]
    outs = [empty_at(m * es, TORCH_DTYPE[dtype], (shift + j * m * es) % 16) for j in range(P)]
    with group(P) as g:
        dt.dt_reduce_scatter(g, dt.DT_ALL_RANKS, [v for _, v in ins], [v for _, v in outs], m, dtype, op)
        torch.cuda.synchronize()
    for j, (gd, v) in enumerate(outs):
        assert_same(host(v), want[j], f"shard {j}")
        assert gd.intact(), f"guard of shard {j}"


# ----------------------------------------------------------------- copies
@pytest.mark.parametrize("layout", ["shared_offset", "mixed", "outputs_apart"])
@pytest.mark.parametrize("row_bytes", [8192, 16, 12, 7, 8190])
@pytest.mark.parametrize("P", [2, 4, 16])
@pytest.mark.parametrize("shared", [False, True])
def test_all_gather_offsets(dt, layout, row_bytes, P, shared):
    # shared_offset: shards and outputs 2 bytes past a boundary; mixed:
    # shards 2 bytes past, outputs aligned; outputs_apart: every output at
    # its own offset (each destination shifted on its own pass)
    rng = np.random.default_rng(row_bytes + P)
    rows = [int(r) for r in rng.integers(0, 300, P)]
    rows[0] = max(rows[0], 1)
    shards = [torch.randint(0, 256, (r * row_bytes,), dtype=torch.uint8, device="cuda") for r in rows]
    want = oracle.all_gather_one([host(x) for x in shards], rows, row_bytes)
    total = sum(rows) * row_bytes
    in_shift = 2
    out_shift = in_shift if layout == "shared_offset" else 0
    ins = [placed(x, in_shift) for x in shards]
    nout = 1 if shared else P
    outs = [empty_at(total, torch.uint8, (out_shift + 3 * q) % 16 if layout == "outputs_apart" else out_shift)
            for q in range(nout)]
    out_views = [outs[0][1]] * P if shared else [v for _, v in outs]
    with group(P) as g:
        dt.dt_all_gather(g, dt.DT_ALL_RANKS, [v for _, v in ins], out_views, rows, 0, row_bytes,
                         flags=dt.DT_SHARED_OUTPUT if shared else 0)
        torch.cuda.synchronize()
    for q, (gd, v) in enumerate(outs):
        assert_same(host(v), want, f"rank {q}")
        assert gd.intact(), f"guard of rank {q}"


@pytest.mark.parametrize("chunk_bytes", [65_536, 1_000_006, 4_096 + 2, 30])
@pytest.mark.parametrize("shifts", [(2, 2), (6, 6), (0, 2), (4, 0), (1, 3)])
@pytest.mark.parametrize("P", [2, 8])
def test_all_to_all_offsets(dt, chunk_bytes, shifts, P):
    # equal shifts with whole-vector chunks share one offset; anything else
    # (unequal shifts, chunks that are not whole vectors) is mixed
    xs = [torch.randint(0, 256, (P * chunk_bytes,), dtype=torch.uint8, device="cuda") for _ in range(P)]
    want = oracle.all_to_all([host(x) for x in xs])
    ins = [placed(x, shifts[0]) for x in xs]
    outs = [empty_at(P * chunk_bytes, torch.uint8, shifts[1]) for _ in range(P)]
    with group(P) as g:
        dt.dt_all_to_all(g, dt.DT_ALL_RANKS, [v for _, v in ins], [v for _, v in outs], chunk_bytes)
        torch.cuda.synchronize()
    for j, (gd, v) in enumerate(outs):
        assert_same(host(v), want[j], f"rank {j}")
        assert gd.intact(), f"guard of rank {j}"


@pytest.mark.parametrize("shifts", [(2, 2), (0, 10)])
def test_replicate_to_shard_and_gather_into_vec_offsets(dt, shifts):
    P, rows, row_bytes = 4, 64, 2 * 1000 + 6
    xs = [torch.randint(0, 256, (rows * row_bytes,), dtype=torch.uint8, device="cuda") for _ in range(P)]
    want = oracle.replicate_to_shard([host(x) for x in xs], rows, row_bytes)
    ins = [placed(x, shifts[0]) for x in xs]
    outs = [empty_at(rows // P * row_bytes, torch.uint8, shifts[1]) for _ in range(P)]
    with group(P) as g:
        dt.dt_replicate_to_shard(g, dt.DT_ALL_RANKS, [v for _, v in ins], [v for _, v in outs], None,
                                 rows, row_bytes)
        torch.cuda.synchronize()
        for r, (gd, v) in enumerate(outs):
            assert_same(host(v), want[r], f"shard {r}")
            assert gd.intact()
        # gather the shards back into a vector of per-rank entries
        srows = [rows // P] * P
        vwant = oracle.all_gather_into_vec([host(v) for _, v in outs], srows, row_bytes)
        vec = [empty_at(rows // P * row_bytes, torch.uint8, shifts[0]) for _ in range(P * P)]
        dt.dt_all_gather_into_vec(g, dt.DT_ALL_RANKS, [v for _, v in outs], [v for _, v in vec],
                                  srows, 0, row_bytes)
        torch.cuda.synchronize()
    for i, (gd, v) in enumerate(vec):
        assert_same(host(v), vwant[i], f"entry {i}")
        assert gd.intact()


def test_rs_ag_step_on_views_two_bytes_past_a_boundary(dt):
    # the bench step (barrier, ReduceScatter AVG, barrier, AllGather) on bf16
    # views that all start 2 bytes past a 16-byte boundary, at 1/16 of the
    # workload's rows
    P, rows, cols = 4, 512, 4096
    g0 = torch.Generator().manual_seed(1)
    xs = [torch.randn(rows, cols, generator=g0).to(torch.bfloat16).cuda() for _ in range(P)]
    snap = [host(x).copy() for x in xs]
    want_rs = oracle.reduce_scatter("bf16", "avg", snap)
    want_ag = oracle.all_gather(want_rs)
    m = rows // P * cols
    ins = [placed(x, 2) for x in xs]
    rs = [empty_at(m * 2, torch.bfloat16, 2) for _ in range(P)]
    ag = [empty_at(rows * cols * 2, torch.bfloat16, 2) for _ in range(P)]
    with group(P) as g:
        dt.dt_barrier(g)
        dt.dt_reduce_scatter(g, dt.DT_ALL_RANKS, [v for _, v in ins], [v for _, v in rs], m, "bf16", "avg")
        dt.dt_barrier(g)
        dt.dt_all_gather(g, dt.DT_ALL_RANKS, [v for _, v in rs], [v for _, v in ag], None, rows // P,
                         cols * 2)
        torch.cuda.synchronize()
    for r in range(P):
        assert_same(host(rs[r][1]), want_rs[r], f"rs {r}")
        assert_same(host(ag[r][1]), want_ag[r], f"ag {r}")
        assert rs[r][0].intact() and ag[r][0].intact()
