"""ReplicateToShard, AllGatherIntoVec and AllToAll(srcDim, destDim): the
remaining placement conversions of the ThreadGroup interface, group-wide and
rank-local, compared bit for bit with the oracle."""
from __future__ import annotations

import threading

import numpy as np
import pytest
import torch

import oracle
from gpu_util import bytes_of, group, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dt():
    from same_device_collective_gb300 import dt as mod
    assert torch.cuda.is_available()
    return mod


def assert_same(got, want, what):
    assert np.array_equal(bytes_of(got), bytes_of(want)), what


def threads(P, fn):
    errs = [None] * P

    def body(r):
        try:
            fn(r)
        except Exception as e:
            errs[r] = e
    ts = [threading.Thread(target=body, args=(r,)) for r in range(P)]
    for t in ts:
        t.start()
    for t in ts:
        t.join(60)
    assert errs == [None] * P, errs


@pytest.mark.parametrize("P", [1, 2, 4, 8])
@pytest.mark.parametrize("cols", [4096, 7])
def test_replicate_to_shard(dt, P, cols):
    rows = 24 * P
    x = torch.randint(-2 ** 31, 2 ** 31 - 1, (rows, cols), dtype=torch.int32, device="cuda")
    ins = [x.clone() for _ in range(P)]
    outs = [torch.empty(rows // P, cols, dtype=torch.int32, device="cuda") for _ in range(P)]
    shard = [(r + 1) % P for r in range(P)]
    with group(P) as g:
        dt.dt_replicate_to_shard(g, dt.DT_ALL_RANKS, ins, outs, None, rows, cols * 4)
        torch.cuda.synchronize()
        want = oracle.replicate_to_shard([host(t) for t in ins], rows, cols * 4)
        for r in range(P):
            assert_same(host(outs[r]), want[r], f"rank {r}")
        dt.dt_replicate_to_shard(g, dt.DT_ALL_RANKS, ins, outs, shard, rows, cols * 4)
        torch.cuda.synchronize()
        want = oracle.replicate_to_shard([host(t) for t in ins], rows, cols * 4, shard)
        for r in range(P):
            assert_same(host(outs[r]), want[r], f"shard idx rank {r}")
        # rank-local: each thread passes its own shard index
        outs2 = [torch.empty_like(o) for o in outs]
        threads(P, lambda r: dt.dt_replicate_to_shard(g, r, [ins[r]], [outs2[r]], [shard[r]], rows,
                                                      cols * 4, torch.cuda.Stream()))
        torch.cuda.synchronize()
        for r in range(P):
            assert_same(host(outs2[r]), want[r], f"rank-local rank {r}")


@pytest.mark.parametrize("P", [1, 2, 3, 8])
@pytest.mark.parametrize("row_bytes", [64, 6])
def test_all_gather_into_vec(dt, P, row_bytes):
    rows = [2 + 3 * r for r in range(P)]
    xs = [torch.randint(0, 256, (rows[r] * row_bytes,), dtype=torch.uint8, device="cuda")
          for r in range(P)]
    vec = [torch.empty(rows[r] * row_bytes, dtype=torch.uint8, device="cuda")
           for q in range(P) for r in range(P)]
    with group(P) as g:
        dt.dt_all_gather_into_vec(g, dt.DT_ALL_RANKS, xs, vec, rows, 0, row_bytes)
        torch.cuda.synchronize()
        want = oracle.all_gather_into_vec([host(x) for x in xs], rows, row_bytes)
        for k in range(P * P):
            assert_same(host(vec[k]), want[k], f"entry {k}")
        vec2 = [torch.empty_like(v) for v in vec]
        threads(P, lambda q: dt.dt_all_gather_into_vec(g, q, [xs[q]], vec2[q * P:(q + 1) * P], None,
                                                       rows[q], row_bytes, torch.cuda.Stream()))
        torch.cuda.synchronize()
        for k in range(P * P):
            assert_same(host(vec2[k]), want[k], f"rank-local entry {k}")


@pytest.mark.parametrize("P", [1, 2, 4, 8])
@pytest.mark.parametrize("src_dim,dest_dim", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.int32])
def test_all_to_all_2d(dt, P, src_dim, dest_dim, dtype):
    R, C = 64 * P, 96 * P
    es = 2 if dtype == torch.bfloat16 else 4
    gen = torch.Generator(device="cuda").manual_seed(P * 10 + src_dim * 2 + dest_dim)
    xs = [torch.randint(-30000, 30000, (R, C), generator=gen, device="cuda").to(dtype)
          for _ in range(P)]
    h = R // P if dest_dim == 0 else R
    w = C // P if dest_dim == 1 else C
    shape = (P * h, w) if src_dim == 0 else (h, P * w)
    outs = [torch.empty(shape, dtype=dtype, device="cuda") for _ in range(P)]
    back = [torch.empty(R, C, dtype=dtype, device="cuda") for _ in range(P)]
    with group(P) as g:
        dt.dt_all_to_all_2d(g, dt.DT_ALL_RANKS, xs, outs, R, C, es, src_dim, dest_dim)
        # and back: S(dest) -> S(src) on the outputs
        dt.dt_all_to_all_2d(g, dt.DT_ALL_RANKS, outs, back, shape[0], shape[1], es, dest_dim, src_dim)
        torch.cuda.synchronize()
        npd = np.int16 if dtype == torch.bfloat16 else np.int32
        want = oracle.all_to_all_2d([host(x).view(npd).reshape(R, C) for x in xs], src_dim, dest_dim)
        for j in range(P):
            assert_same(host(outs[j]), want[j], f"rank {j}")
            assert torch.equal(back[j].view(torch.int16 if es == 2 else torch.int32),
                               xs[j].view(torch.int16 if es == 2 else torch.int32)), f"round trip {j}"
        outs2 = [torch.empty_like(o) for o in outs]
        threads(P, lambda r: dt.dt_all_to_all_2d(g, r, [xs[r]], [outs2[r]], R, C, es, src_dim,
                                                 dest_dim, torch.cuda.Stream()))
        torch.cuda.synchronize()
        for j in range(P):
            assert_same(host(outs2[j]), want[j], f"rank-local rank {j}")


def test_all_to_all_2d_odd_widths_take_the_byte_path(dt):
    P, R, C = 2, 6, 10                      # C / P * 2 bytes = 10: not a 16-byte multiple
    xs = [torch.randint(0, 1000, (R, C), device="cuda").to(torch.bfloat16) for _ in range(P)]
    outs = [torch.empty(P * R, C // P, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    with group(P) as g:
        dt.dt_all_to_all_2d(g, dt.DT_ALL_RANKS, xs, outs, R, C, 2, 0, 1)
        torch.cuda.synchronize()
    want = oracle.all_to_all_2d([host(x).view(np.int16).reshape(R, C) for x in xs], 0, 1)
    for j in range(P):
        assert_same(host(outs[j]), want[j], f"rank {j}")


def test_placement_argument_errors(dt):
    P = 2
    x = [torch.zeros(8, 8, device="cuda") for _ in range(P)]
    o = [torch.zeros(8, 8, device="cuda") for _ in range(P)]
    with group(P) as g:
        n0 = dt.dt_launch_count()
        with pytest.raises(dt.DtError):          # rows not a multiple of P
            dt.dt_replicate_to_shard(g, dt.DT_ALL_RANKS, x, o, None, 7, 32)
        with pytest.raises(dt.DtError):          # shard index out of range
            dt.dt_replicate_to_shard(g, dt.DT_ALL_RANKS, x, o, [0, 5], 8, 32)
        with pytest.raises(dt.DtError):          # C not a multiple of P for dest_dim 1
            dt.dt_all_to_all_2d(g, dt.DT_ALL_RANKS, x, o, 8, 7, 4, 0, 1)
        with pytest.raises(dt.DtError):          # bad dim
            dt.dt_all_to_all_2d(g, dt.DT_ALL_RANKS, x, o, 8, 8, 4, 2, 0)
        with pytest.raises(dt.DtError):          # output overlaps an input
            dt.dt_all_gather_into_vec(g, dt.DT_ALL_RANKS, x, [o[0], o[1], x[0], o[1]], None, 1, 32)
        assert dt.dt_launch_count() == n0
