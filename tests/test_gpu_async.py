"""Async work handles and the pipelined ReduceScatter -> AllReduce schedule.

The async scope follows the async mode of the PyTorch page (§四.3): work runs
on the group's own stream after it waits for the caller's stream, and the
caller later waits on the work's end event.  The pipeline test replays the
post_backward schedule of the hyper-parallel issue ("异步融合 AllReduce 流水线
优化"): for each module, wait for the previous module's ReduceScatter, issue
this module's ReduceScatter, issue the previous module's fused AllReduce, and
at the root hook wait for every AllReduce; it runs on a 2 x 2 mesh of logical
ranks (shard groups {0,1}, {2,3}; replicate groups {0,2}, {1,3}) and must give
exactly the sequential result."""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import oracle
from gpu_util import bytes_of, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dt():
    from same_device_collective_gb300 import dt as mod
    assert torch.cuda.is_available()
    return mod


def test_async_scope_allreduce_and_work_handles(dt):
    P, n = 4, 1 << 20
    xs = [torch.randn(n, device="cuda") for _ in range(P)]
    outs = [torch.empty_like(x) for x in xs]
    caller = torch.cuda.Stream()
    other = torch.cuda.Stream()
    g = dt.dt_group_create(P, 0)
    try:
        with torch.cuda.stream(caller):
            ys = [x * 2 for x in xs]          # produced on the caller's stream
            cs = dt.dt_async_begin(g, caller)
            assert cs != caller.cuda_stream
            dt.dt_allreduce(g, dt.DT_ALL_RANKS, ys, outs, n, "f32", "sum", 0, cs)
            w = dt.dt_async_end(g)
        dt.dt_work_wait(w, other)
        with torch.cuda.stream(other):
            got = [o.clone() for o in outs]   # read after the work, on another stream
        deadline = time.time() + 10
        while dt.dt_work_query(w) == dt.DT_NOT_READY and time.time() < deadline:
            time.sleep(0.001)
        assert dt.dt_work_query(w) == dt.DT_OK
        dt.dt_work_free(w)
        torch.cuda.synchronize()
        want = oracle.allreduce("f32", "sum", [host(y) for y in ys])
        for q in range(P):
            assert np.array_equal(bytes_of(host(got[q])), bytes_of(want[q]))
    finally:
        torch.cuda.synchronize()
        dt.dt_group_destroy(g)


def test_async_scope_errors(dt):
    g = dt.dt_group_create(2, 0)
    try:
        with pytest.raises(dt.DtError):
            dt.dt_async_end(g)                # no open scope
        dt.dt_async_begin(g)
        with pytest.raises(dt.DtError):
            dt.dt_async_begin(g)              # one scope at a time
        w = dt.dt_async_end(g)                # an empty scope is a valid work
        dt.dt_work_wait(w)
        torch.cuda.synchronize()
        assert dt.dt_work_query(w) == dt.DT_OK
        dt.dt_work_free(w)
    finally:
        dt.dt_group_destroy(g)


def hsdp_mesh(dt):
    shard = [dt.dt_group_create(2, 0), dt.dt_group_create(2, 0)]      # {0,1}, {2,3}
    repl = [dt.dt_group_create(2, 0), dt.dt_group_create(2, 0)]       # {0,2}, {1,3}
    return shard, repl


def run_pipeline(dt, shard, repl, grads, rs, fin, n, compute):
    """The post_backward schedule; returns nothing, results land in fin."""
    M = len(grads)
    prev_rs = []
    pending_ar = []
    ALL = dt.DT_ALL_RANKS

    def issue_rs(m):
        works = []
        for s in range(2):
            cs = dt.dt_async_begin(shard[s], compute)
            a, b = 2 * s, 2 * s + 1
            dt.dt_reduce_scatter(shard[s], ALL, [grads[m][a], grads[m][b]], [rs[m][a], rs[m][b]],
                                 n // 2, "bf16", "avg", cs)
            works.append(dt.dt_async_end(shard[s]))
        return works

    def issue_ar(m):
        for k in range(2):
            cs = dt.dt_async_begin(repl[k], compute)
            a, b = k, k + 2
            dt.dt_allreduce(repl[k], ALL, [rs[m][a], rs[m][b]], [fin[m][a], fin[m][b]], n // 2,
                            "bf16", "avg", 0, cs)
            pending_ar.append(dt.dt_async_end(repl[k]))

    for m in range(M):
        for w in prev_rs:                       # 1. wait the previous ReduceScatter
            dt.dt_work_wait(w, compute)
            dt.dt_work_free(w)
        cur = issue_rs(m)                       # 2. issue this module's ReduceScatter
        if m > 0:
            issue_ar(m - 1)                     # 3. issue the previous module's AllReduce
        prev_rs = cur
    for w in prev_rs:                           # root hook: the last module ...
        dt.dt_work_wait(w, compute)
        dt.dt_work_free(w)
    issue_ar(M - 1)
    for w in pending_ar:                        # ... then wait every AllReduce
        dt.dt_work_wait(w, compute)
        dt.dt_work_free(w)


def test_hsdp_pipeline_equals_sequential_oracle(dt):
    M, n = 5, 3 * 4096 * 2
    gen = torch.Generator(device="cuda").manual_seed(9)
    grads = [[torch.randn(n, generator=gen, device="cuda").to(torch.bfloat16) for _ in range(4)]
             for _ in range(M)]
    rs = [[torch.empty(n // 2, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
          for _ in range(M)]
    fin = [[torch.empty(n // 2, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
           for _ in range(M)]
    shard, repl = hsdp_mesh(dt)
    compute = torch.cuda.Stream()
    try:
        run_pipeline(dt, shard, repl, grads, rs, fin, n, compute)
        torch.cuda.synchronize()
        for m in range(M):
            h = [host(x) for x in grads[m]]
            r = oracle.reduce_scatter("bf16", "avg", h[0:2]) + oracle.reduce_scatter("bf16", "avg", h[2:4])
            for k in range(2):
                want = oracle.allreduce("bf16", "avg", [r[k], r[k + 2]])
                assert np.array_equal(host(fin[m][k]), want[0]), (m, k)
                assert np.array_equal(host(fin[m][k + 2]), want[1]), (m, k + 2)
        for g in shard + repl:
            assert dt.dt_group_check(g) == dt.DT_OK
    finally:
        torch.cuda.synchronize()
        for g in shard + repl:
            dt.dt_group_destroy(g)
