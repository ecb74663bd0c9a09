"""Parity at the workloads' full sizes, launched the way bench.py launches them.

Where the oracle can take the whole problem on the host it does (the P=2
AllReduce, the RS+AG step, the bucket all-reduce, the uneven gather's single
concatenation); where the problem is many GiB the
check uses outputs the oracle computes one by one (sampled element positions
of a reduction) plus properties that hold at any size (all-to-all twice is
the identity; every per-rank gather output equals the shared one).  The
8-rank all-to-all of 512 MiB per rank is compared with the oracle on every
byte.  All comparisons are bit-exact.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import ELEM, TORCH_DTYPE, bytes_of, group, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dt():
    from same_device_collective_gb300 import dt as mod
    assert torch.cuda.is_available()
    return mod


@pytest.fixture(scope="module")
def wl():
    from same_device_collective_gb300 import workloads
    return workloads


def assert_same(got, want, what):
    g, w = bytes_of(got), bytes_of(want)
    assert g.size == w.size, what
    if not np.array_equal(g, w):
        bad = np.nonzero(g != w)[0]
        raise AssertionError(f"{what}: {bad.size} bytes differ, first at byte {bad[0]}")


def sample_reduce(dtype, op, ins, out, in_off, n, k=4096, seed=0):
    """Compare `out[i]` with the oracle's reduction of ins[r][in_off + i] at k
    sampled positions i < n."""
    g = torch.Generator(device=ins[0].device).manual_seed(seed)
    idx = torch.randint(0, n, (k,), generator=g, device=ins[0].device)
    cols = [host(x.reshape(-1)[idx + in_off]) for x in ins]
    want = oracle.reduce(dtype, op, cols)
    got = host(out.reshape(-1)[idx])
    assert_same(got, want, f"sampled {dtype} {op}")


# ------------------------------------------------------- the full workloads
def test_full_allreduce_sum_f32_P2_n2e20(dt, wl):
    w = wl.allreduce_small()
    xs = [x.cuda() for x in w.inputs]
    outs = [torch.empty_like(x) for x in xs]
    with group(2) as g:
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, outs, xs[0].numel(), "f32", "sum")
        torch.cuda.synchronize()
    want = oracle.allreduce("f32", "sum", [host(x) for x in w.inputs])
    for q in range(2):
        assert_same(host(outs[q]), want[q], f"rank {q}")


def test_full_rs_avg_then_ag_bf16_P4_8192x4096(dt, wl):
    P, R, C = 4, 8192, 4096
    w = wl.rs_ag(device="cuda")
    xs = w.inputs
    m = R // P * C
    rs = [torch.empty(R // P, C, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    ag = [torch.empty(R, C, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    with group(P) as g:                      # the bench's step, twice
        for _ in range(2):
            dt.dt_barrier(g)
            dt.dt_reduce_scatter(g, dt.DT_ALL_RANKS, xs, rs, m, "bf16", "avg")
            dt.dt_barrier(g)
            dt.dt_all_gather(g, dt.DT_ALL_RANKS, rs, ag, None, R // P, C * 2)
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
        assert np.array_equal(dt.dt_debug_read_window(g), oracle.expected_window(P, 4))
    want_rs = oracle.reduce_scatter("bf16", "avg", [host(x) for x in xs])
    for r in range(P):
        assert_same(host(rs[r]), want_rs[r], f"reduce_scatter rank {r}")
    want_ag = oracle.all_gather_one(want_rs, [1] * P, m * 2)
    for q in range(P):
        assert_same(host(ag[q]), want_ag, f"all_gather rank {q}")


def test_full_bucket_allreduce_avg_bf16_P8_T200(dt, wl):
    P = 8
    w = wl.bucket_grads(device="cuda")
    counts = w.meta["counts"]
    ref = [[host(x).copy() for x in row] for row in w.inputs]
    _, nb = dt.dt_bucket_plan(counts, 2, wl.BUCKET_CAP_BYTES)
    # the argument form the bench times: a prepared pointer table
    table, cnt = dt.pointer_table(w.inputs), np.asarray(counts, dtype=np.uint64)
    with group(P) as g:
        dt.dt_bucket_allreduce(g, table, cnt, "bf16", "avg", wl.BUCKET_CAP_BYTES)
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
        assert np.array_equal(dt.dt_debug_read_window(g), oracle.expected_window(P, nb - 1))
    oracle.bucket_allreduce("bf16", "avg", ref)
    for t in range(len(counts)):
        for p in range(P):
            assert_same(host(w.inputs[t][p]), ref[t][p], f"tensor {t} rank {p}")


def test_full_all_to_all_bf16_P8_65536x4096(dt, wl):
    P = 8
    w = wl.all_to_all_tokens(device="cuda")
    xs = w.inputs
    outs = [torch.empty_like(x) for x in xs]
    back = [torch.empty_like(x) for x in xs]
    c = xs[0].numel() // P                    # elements per chunk
    with group(P) as g:
        dt.dt_all_to_all(g, dt.DT_ALL_RANKS, xs, outs, c * 2)
        dt.dt_all_to_all(g, dt.DT_ALL_RANKS, outs, back, c * 2)
        torch.cuda.synchronize()
    for x, b in zip(xs, back):
        assert torch.equal(x.view(torch.int16), b.view(torch.int16))   # twice = identity
    del back
    # every byte: the oracle's all-to-all of the inputs read back from the
    # device (4 GiB), compared one destination rank (512 MiB) at a time.  At
    # this size each rank streams more than L2 holds, so the launch takes the
    # 16 KiB x 12 single-destination tile shape.
    want = oracle.all_to_all([host(x) for x in xs])
    for j in range(P):
        assert_same(host(outs[j]), want[j], f"rank {j}")
        want[j] = None


def test_full_uneven_all_gather_i32_P8_rows16384(dt, wl):
    P = 8
    w = wl.uneven_gather(device="cuda")
    rows, cols = w.meta["rows"], w.meta["cols"]
    total = sum(rows)
    shared = torch.empty(total, cols, dtype=torch.int32, device="cuda")
    per = [torch.empty(total, cols, dtype=torch.int32, device="cuda") for _ in range(P)]
    with group(P) as g:
        dt.dt_all_gather(g, dt.DT_ALL_RANKS, w.inputs, [shared] * P, rows, 0, cols * 4,
                         flags=dt.DT_SHARED_OUTPUT)
        dt.dt_all_gather(g, dt.DT_ALL_RANKS, w.inputs, per, rows, 0, cols * 4)
        torch.cuda.synchronize()
    want = oracle.all_gather_one([host(x) for x in w.inputs], rows, cols * 4)
    assert_same(host(shared), want, "shared output")
    for q in range(P):
        assert torch.equal(per[q], shared), f"rank {q}"


# ------------------------------------------- size sweep 4 KiB .. 1 GiB per rank
SWEEP_SMALL = [4096, 1 << 20]


@pytest.mark.parametrize("P", [2, 4, 8, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "max"])
def test_sweep_reductions_small_sizes(dt, wl, P, dtype, op):
    sizes = SWEEP_SMALL + ([16 << 20] if P in (2, 16) else [])
    for nbytes in sizes:
        w = wl.sweep_inputs(4, P, nbytes, dtype, device="cuda")
        xs = w.inputs
        n = xs[0].numel()
        outs = [torch.empty_like(x) for x in xs]
        m = n // P
        rs = [torch.empty(m, dtype=TORCH_DTYPE[dtype], device="cuda") for _ in range(P)]
        with group(P) as g:
            dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, outs, n, dtype, op)
            dt.dt_reduce_scatter(g, dt.DT_ALL_RANKS, xs, rs, m, dtype, op)
            torch.cuda.synchronize()
        hx = [host(x) for x in xs]
        want = oracle.allreduce(dtype, op, hx)
        for q in range(P):
            assert_same(host(outs[q]), want[q], f"AR {nbytes} B rank {q}")
        want = oracle.reduce_scatter(dtype, op, hx)
        for r in range(P):
            assert_same(host(rs[r]), want[r], f"RS {nbytes} B rank {r}")


@pytest.mark.parametrize("P", [2, 4, 8, 16])
def test_sweep_copies_small_sizes(dt, wl, P):
    for nbytes in SWEEP_SMALL + [16 << 20]:
        w = wl.sweep_inputs(4, P, nbytes, "i32", device="cuda")
        xs = w.inputs
        ag = [torch.empty(P * xs[0].numel(), dtype=torch.int32, device="cuda") for _ in range(P)]
        a2a = [torch.empty_like(x) for x in xs]
        with group(P) as g:
            dt.dt_all_gather(g, dt.DT_ALL_RANKS, xs, ag, None, 1, nbytes)
            dt.dt_all_to_all(g, dt.DT_ALL_RANKS, xs, a2a, nbytes // P)
            torch.cuda.synchronize()
        hx = [host(x) for x in xs]
        want = oracle.all_gather_one(hx, [1] * P, nbytes)
        for q in range(P):
            assert_same(host(ag[q]), want, f"AG {nbytes} B rank {q}")
        want = oracle.all_to_all(hx)
        for j in range(P):
            assert_same(host(a2a[j]), want[j], f"A2A {nbytes} B rank {j}")


def test_sweep_large_reductions_sampled(dt, wl):
    # AllReduce fp32 sum, P=16, 256 MiB per rank; ReduceScatter bf16 max, P=8, 1 GiB per rank
    P = 16
    w = wl.sweep_inputs(4, P, 256 << 20, "f32", device="cuda")
    outs = [torch.empty_like(x) for x in w.inputs]
    n = w.inputs[0].numel()
    with group(P) as g:
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, w.inputs, outs, n, "f32", "sum")
        torch.cuda.synchronize()
    for q in (0, 7, 15):
        sample_reduce("f32", "sum", w.inputs, outs[q], 0, n, seed=q)
    del w, outs
    P = 8
    w = wl.sweep_inputs(4, P, 1 << 30, "bf16", device="cuda")
    n = w.inputs[0].numel()
    m = n // P
    rs = [torch.empty(m, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    with group(P) as g:
        dt.dt_reduce_scatter(g, dt.DT_ALL_RANKS, w.inputs, rs, m, "bf16", "max")
        torch.cuda.synchronize()
    for r in (0, 3, 7):
        sample_reduce("bf16", "max", w.inputs, rs[r], r * m, m, seed=r)
    del w, rs
    torch.cuda.empty_cache()


def test_sweep_large_copies_sampled(dt, wl):
    P = 16
    w = wl.sweep_inputs(4, P, 256 << 20, "i32", device="cuda")
    xs = w.inputs
    shared = torch.empty(P * xs[0].numel(), dtype=torch.int32, device="cuda")
    a2a = [torch.empty_like(x) for x in xs]
    back = [torch.empty_like(x) for x in xs]
    with group(P) as g:
        dt.dt_all_gather(g, dt.DT_ALL_RANKS, xs, [shared] * P, None, 1, 256 << 20,
                         flags=dt.DT_SHARED_OUTPUT)
        dt.dt_all_to_all(g, dt.DT_ALL_RANKS, xs, a2a, (256 << 20) // P)
        dt.dt_all_to_all(g, dt.DT_ALL_RANKS, a2a, back, (256 << 20) // P)
        torch.cuda.synchronize()
    for x, b in zip(xs, back):
        assert torch.equal(x, b)                       # all-to-all twice = identity
    # sampled positions k of every shard: the oracle's gather of the sampled
    # shards must equal the gathered output at r * n + k
    n = xs[0].numel()
    gen = torch.Generator(device="cuda").manual_seed(5)
    k = torch.randint(0, n, (4096,), generator=gen, device="cuda")
    want = oracle.all_gather_one([host(x[k]) for x in xs], [1] * P, 4096 * 4)
    idx = (torch.arange(P, device="cuda")[:, None] * n + k[None, :]).reshape(-1)
    assert_same(host(shared[idx]), want, "shared gather, sampled")
    c = n // P
    kc = k % c
    idx = (torch.arange(P, device="cuda")[:, None] * c + kc[None, :]).reshape(-1)
    want = oracle.all_to_all([host(x[idx]) for x in xs])
    for j in range(P):
        assert_same(host(a2a[j][idx]), want[j], f"all_to_all sampled rank {j}")
    del w, xs, shared, a2a, back
    torch.cuda.empty_cache()


def test_barrier_1e5_calls_P16(dt):
    P, calls = 16, 100_000
    with group(P) as g:
        s = torch.cuda.current_stream().cuda_stream
        for _ in range(calls):
            dt.dt_barrier(g, dt.DT_ALL_RANKS, s)
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
        assert np.array_equal(dt.dt_debug_read_window(g), oracle.expected_window(P, calls))
