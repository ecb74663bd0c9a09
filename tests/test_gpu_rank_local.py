"""Rank-local calls: P host threads, one per rank, each with its own buffers
and its own CUDA stream, as DTorch drives ThreadGroup (one thread per rank,
meeting through the MemoryTensorStore).  Results are compared bit for bit with
the oracle; the host rendezvous's failure path (a rank that never arrives) is
checked through its time limit, with no GPU fault."""
from __future__ import annotations

import threading

import numpy as np
import pytest
import torch

import oracle
from gpu_util import TORCH_DTYPE, bytes_of, group, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dt():
    from same_device_collective_gb300 import dt as mod
    assert torch.cuda.is_available()
    return mod


def run_ranks(P, fn):
    """Run fn(rank) on P threads; returns the list of exceptions (None = ok)."""
    errs = [None] * P

    def body(r):
        try:
            fn(r)
        except Exception as e:   # collected and checked by the caller
            errs[r] = e

    ts = [threading.Thread(target=body, args=(r,)) for r in range(P)]
    for t in ts:
        t.start()
    for t in ts:
        t.join(60)
    assert not any(t.is_alive() for t in ts)
    return errs


def assert_same(got, want, what):
    assert np.array_equal(bytes_of(got), bytes_of(want)), what


@pytest.mark.parametrize("P", [2, 4, 8])
@pytest.mark.parametrize("dtype,op", [("f32", "sum"), ("bf16", "avg"), ("i32", "max")])
def test_rank_local_allreduce_and_reduce_scatter(dt, P, dtype, op):
    n = 4096 * P + 8 * P
    m = n // P
    streams = [torch.cuda.Stream() for _ in range(P)]
    ins = [None] * P
    outs = [None] * P
    rss = [None] * P
    with group(P) as g:
        def rank(r):
            s = streams[r]
            with torch.cuda.stream(s):
                gen = torch.Generator(device="cuda").manual_seed(1000 + r)
                if dtype == "i32":
                    x = torch.randint(-2 ** 20, 2 ** 20, (n,), generator=gen, device="cuda",
                                      dtype=torch.int32)
                else:
                    x = (torch.rand(n, generator=gen, device="cuda") * 2 - 1).to(TORCH_DTYPE[dtype])
                o = torch.empty_like(x)
                rs = torch.empty(m, dtype=x.dtype, device="cuda")
                # inputs were produced on this rank's stream just before the call
                dt.dt_allreduce(g, r, [x], [o], n, dtype, op, 0, s)
                dt.dt_reduce_scatter(g, r, [x], [rs], m, dtype, op, s)
                ins[r], outs[r], rss[r] = x, o.clone(), rs.clone()   # read back in stream order
        errs = run_ranks(P, rank)
        assert errs == [None] * P, errs
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
    hx = [host(x) for x in ins]
    want = oracle.allreduce(dtype, op, hx)
    for q in range(P):
        assert_same(host(outs[q]), want[q], f"allreduce rank {q}")
    want = oracle.reduce_scatter(dtype, op, hx)
    for r in range(P):
        assert_same(host(rss[r]), want[r], f"reduce_scatter rank {r}")


@pytest.mark.parametrize("P", [2, 3, 8])
def test_rank_local_uneven_all_gather_and_all_to_all(dt, P):
    row_bytes = 64
    rows = [3 + 5 * r for r in range(P)]
    total = sum(rows)
    chunk = 256
    streams = [torch.cuda.Stream() for _ in range(P)]
    xs = [torch.randint(0, 256, (rows[r] * row_bytes,), dtype=torch.uint8, device="cuda")
          for r in range(P)]
    a2a_in = [torch.randint(0, 256, (P * chunk,), dtype=torch.uint8, device="cuda")
              for _ in range(P)]
    torch.cuda.synchronize()
    ag = [torch.empty(total * row_bytes, dtype=torch.uint8, device="cuda") for _ in range(P)]
    a2a = [torch.empty(P * chunk, dtype=torch.uint8, device="cuda") for _ in range(P)]
    with group(P) as g:
        def rank(r):
            s = streams[r]
            dt.dt_all_gather(g, r, [xs[r]], [ag[r]], None, rows[r], row_bytes, 0, s)
            dt.dt_all_to_all(g, r, [a2a_in[r]], [a2a[r]], chunk, s)
        errs = run_ranks(P, rank)
        assert errs == [None] * P, errs
        torch.cuda.synchronize()
    want = oracle.all_gather_one([host(x) for x in xs], rows, row_bytes)
    for q in range(P):
        assert_same(host(ag[q]), want, f"all_gather rank {q}")
    want = oracle.all_to_all([host(x) for x in a2a_in])
    for j in range(P):
        assert_same(host(a2a[j]), want[j], f"all_to_all rank {j}")


@pytest.mark.parametrize("P", [2, 4, 16])
def test_rank_local_barrier_window(dt, P):
    G = 5
    streams = [torch.cuda.Stream() for _ in range(P)]
    with group(P) as g:
        def rank(r):
            for _ in range(G):
                dt.dt_barrier(g, r, streams[r])
        errs = run_ranks(P, rank)
        assert errs == [None] * P, errs
        torch.cuda.synchronize()
        assert np.array_equal(dt.dt_debug_read_window(g), oracle.expected_window(P, G))
        assert dt.dt_group_check(g) == dt.DT_OK


def test_rank_local_mismatched_calls_are_rejected(dt):
    P = 3
    xs = [torch.ones(64, device="cuda") for _ in range(P)]
    os_ = [torch.empty(64, device="cuda") for _ in range(P)]
    with group(P) as g:
        n0 = dt.dt_launch_count()

        def rank(r):
            n = 64 if r != 1 else 32      # rank 1 disagrees on the size
            dt.dt_allreduce(g, r, [xs[r]], [os_[r]], n, "f32", "sum", 0,
                            torch.cuda.current_stream())
        errs = run_ranks(P, rank)
        assert all(isinstance(e, dt.DtError) and e.status == dt.DT_ERR_INVALID for e in errs)
        assert dt.dt_launch_count() == n0
        assert dt.dt_group_check(g) == dt.DT_OK


def test_rank_local_missing_rank_times_out_and_reset_recovers(dt):
    P = 4
    streams = [torch.cuda.Stream() for _ in range(P)]
    with group(P) as g:
        dt.dt_group_set_timeout_ms(g, 300)
        n0 = dt.dt_launch_count()

        def rank(r):
            if r == 2:
                return                       # this rank never arrives
            dt.dt_barrier(g, r, streams[r])
        errs = run_ranks(P, rank)
        for r in range(P):
            if r == 2:
                assert errs[r] is None
            else:
                assert isinstance(errs[r], dt.DtError) and errs[r].status == dt.DT_ERR_TIMEOUT
        assert dt.dt_launch_count() == n0   # nothing was launched
        assert dt.dt_group_check(g) == dt.DT_ERR_TIMEOUT
        with pytest.raises(dt.DtError):
            dt.dt_barrier(g, 2, streams[2])  # the late rank finds the group poisoned
        dt.dt_group_reset(g)
        assert dt.dt_group_check(g) == dt.DT_OK
        errs = run_ranks(P, lambda r: dt.dt_barrier(g, r, streams[r]))
        assert errs == [None] * P, errs
        torch.cuda.synchronize()
        assert np.array_equal(dt.dt_debug_read_window(g), oracle.expected_window(P, 1))


def test_native_thread_driver_runs_the_rank_local_step():
    # rank_local_step (built with the library) runs the barrier / ReduceScatter /
    # barrier / AllGather step from one std::thread per rank through the C ABI;
    # here at a small ragged size, P=3, with a clean group status at the end.
    import json
    import os
    import subprocess
    tool = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "same_device_collective_gb300", "rank_local_step")
    res = subprocess.run([tool, "3", "96", "72", "50"], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr
    out = json.loads(res.stdout.strip().splitlines()[-1])
    assert out["status_ok"] is True and out["P"] == 3 and out["steps"] == 50
    bad = subprocess.run([tool, "3", "97", "72", "5"], capture_output=True, text=True, timeout=60)
    assert bad.returncode != 0 and "error" in json.loads(bad.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("shared_stream", [False, True])
@pytest.mark.parametrize("P", [3, 8])
def test_rank_local_chained_rounds_stay_ordered(dt, P, shared_stream):
    # P threads run the same seeded sequence of 120 rounds.  Each round first
    # updates the rank's buffer on its own stream (b = 0.5 b + (k + r)), then
    # makes one rank-local call on it: an in-place AllReduce, a ReduceScatter
    # (avg) followed by an AllGather back into b, an AllToAll copied back into
    # b, or a bare barrier.  Every input depends on the previous collective's
    # output, so an ordering slip anywhere shows in the final buffers, which a
    # host replica built from the oracle must match bit for bit.  With
    # shared_stream every rank thread uses one stream (the calls then need no
    # cross-stream waits).
    K, n = 120, 24_024
    m = n // P
    rng = np.random.default_rng(P)
    kinds = rng.choice(["ar", "rs_ag", "a2a", "barrier"], size=K, p=[0.35, 0.3, 0.2, 0.15])
    streams = [torch.cuda.Stream() for _ in range(P)]
    if shared_stream:
        streams = [streams[0]] * P
    bufs = [torch.arange(n, dtype=torch.float32, device="cuda") * (r + 1) / n for r in range(P)]
    host_b = [host(b).copy() for b in bufs]
    torch.cuda.synchronize()
    with group(P) as g:
        def rank(r):
            s = streams[r]
            b = bufs[r]
            shard = torch.empty(m, device="cuda")
            tmp = torch.empty(n, device="cuda")
            with torch.cuda.stream(s):
                for k, kind in enumerate(kinds):
                    b.mul_(0.5).add_(float(k + r))
                    if kind == "ar":
                        dt.dt_allreduce(g, r, [b], [b], n, "f32", "sum", 0, s)
                    elif kind == "rs_ag":
                        dt.dt_reduce_scatter(g, r, [b], [shard], m, "f32", "avg", s)
                        dt.dt_all_gather(g, r, [shard], [b], None, m, 4 * 1, 0, s)
                    elif kind == "a2a":
                        dt.dt_all_to_all(g, r, [b], [tmp], m * 4, s)
                        b.copy_(tmp)
                    else:
                        dt.dt_barrier(g, r, s)
        errs = run_ranks(P, rank)
        assert errs == [None] * P, errs
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
        win = dt.dt_debug_read_window(g)
    for k, kind in enumerate(kinds):
        host_b = [(hb * np.float32(0.5)).astype(np.float32) + np.float32(k + r)
                  for r, hb in enumerate(host_b)]
        host_b = [hb.astype(np.float32) for hb in host_b]
        if kind == "ar":
            host_b = oracle.allreduce("f32", "sum", host_b)
        elif kind == "rs_ag":
            rs = oracle.reduce_scatter("f32", "avg", host_b)
            host_b = [g.view(np.float32) for g in oracle.all_gather(rs, [m] * P, 4)]
        elif kind == "a2a":
            host_b = [a.view(np.float32) for a in oracle.all_to_all(host_b)]
    for r in range(P):
        assert_same(host(bufs[r]), host_b[r], f"rank {r}")
    assert np.array_equal(win, oracle.expected_window(P, int((kinds == "barrier").sum())))


def test_prepared_calls_from_rank_threads(dt):
    # The RS(avg) + AG step from four rank threads through prepared calls
    # (arguments marshalled once, the same C call each step), three steps in a
    # row, compared with the oracle; a prepared group-wide AllReduce matches
    # the per-call function bit for bit.
    P, rows, cols = 4, 64, 40
    gen = torch.Generator().manual_seed(77)
    xs = [torch.randn(rows, cols, generator=gen).to(torch.bfloat16).cuda() for _ in range(P)]
    m = rows // P * cols
    rs = [torch.empty(rows // P, cols, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    ag = [torch.empty(rows, cols, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    streams = [torch.cuda.Stream() for _ in range(P)]
    torch.cuda.synchronize()
    with group(P) as g:
        steps = []
        for r in range(P):
            raw = streams[r].cuda_stream
            steps.append([dt.prepare(dt.dt_barrier, g, r, raw),
                          dt.prepare(dt.dt_reduce_scatter, g, r, [xs[r]], [rs[r]], m, "bf16", "avg",
                                     raw),
                          dt.prepare(dt.dt_barrier, g, r, raw),
                          dt.prepare(dt.dt_all_gather, g, r, [rs[r]], [ag[r]], None, rows // P,
                                     cols * 2, 0, raw)])

        def rank(r):
            for _ in range(3):
                for call in steps[r]:
                    call()

        assert run_ranks(P, rank) == [None] * P
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
        want_rs = oracle.reduce_scatter("bf16", "avg", [host(x) for x in xs])
        want_ag = oracle.all_gather(want_rs)
        for r in range(P):
            assert_same(host(rs[r]), want_rs[r], f"reduce_scatter rank {r}")
            assert_same(host(ag[r]), want_ag[r], f"all_gather rank {r}")
        assert np.array_equal(dt.dt_debug_read_window(g), oracle.expected_window(P, 6))

        a = [torch.empty_like(x) for x in xs]
        b = [torch.empty_like(x) for x in xs]
        s = torch.cuda.current_stream().cuda_stream
        dt.prepare(dt.dt_allreduce, g, dt.DT_ALL_RANKS, xs, a, rows * cols, "bf16", "sum", 0, s)()
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, b, rows * cols, "bf16", "sum", 0, s)
        torch.cuda.synchronize()
        for q in range(P):
            assert_same(host(a[q]), host(b[q]), f"allreduce rank {q}")


@pytest.mark.parametrize("P", [2, 4, 8])
def test_rank_local_barrier_orders_data_ring(dt, P):
    # The barrier page's ordering example from rank threads: each rank stages
    # its values on its own stream (after a stream sleep of its own length, so
    # the ranks finish staging at different times), meets the others in a
    # rank-local barrier, then reads the next rank's stage on its own stream.
    # Without the barrier's ordering a rank would read a stale stage.
    n, rounds = 1 << 16, 6
    streams = [torch.cuda.Stream() for _ in range(P)]
    stage = [torch.zeros(n, dtype=torch.int32, device="cuda") for _ in range(P)]
    outs = [[torch.empty(n, dtype=torch.int32, device="cuda") for _ in range(rounds)] for _ in range(P)]
    vals = [[torch.full((n,), 1000 * k + r, dtype=torch.int32, device="cuda") for k in range(rounds)]
            for r in range(P)]
    torch.cuda.synchronize()
    with group(P) as g:
        def rank(r):
            s = streams[r]
            with torch.cuda.stream(s):
                for k in range(rounds):
                    torch.cuda._sleep(200_000 * ((r * 7 + k * 3) % P + 1))
                    stage[r].copy_(vals[r][k])
                    dt.dt_barrier(g, r, s)
                    outs[r][k].copy_(stage[(r + 1) % P])
                    dt.dt_barrier(g, r, s)       # nobody restages before everyone has read
        errs = run_ranks(P, rank)
        assert errs == [None] * P, errs
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
        assert np.array_equal(dt.dt_debug_read_window(g), oracle.expected_window(P, 2 * rounds))
    for r in range(P):
        for k in range(rounds):
            assert torch.all(outs[r][k] == 1000 * k + (r + 1) % P), f"rank {r} round {k}"
