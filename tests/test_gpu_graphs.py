"""Group-wide calls captured in a CUDA graph replay correctly.

The barrier keeps its generation on the device, so every replay advances the
signal window; collectives carry their rank pointers in the kernel parameter
block; a bucket call captured while its plan is cached replays its launches
against that plan.  Each replay runs on fresh input values and is checked
against the oracle, bit for bit.
"""
from __future__ import annotations

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


def test_rs_ag_step_graph_replays(dt):
    P, R, C = 4, 512, 264            # bf16 [512, 264] per rank: several vectors per thread, 528-byte rows
    m = R // P * C
    ALL = dt.DT_ALL_RANKS
    gen = torch.Generator(device="cuda").manual_seed(11)
    xs = [torch.empty(R, C, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    rs = [torch.empty(R // P, C, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    ag = [torch.empty(R, C, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    s = torch.cuda.Stream()
    with group(P) as g:
        def step():
            dt.dt_barrier(g, ALL, s)
            dt.dt_reduce_scatter(g, ALL, xs, rs, m, "bf16", "avg", s)
            dt.dt_barrier(g, ALL, s)
            dt.dt_all_gather(g, ALL, rs, ag, None, R // P, C * 2, 0, s)
        with torch.cuda.stream(s):
            for x in xs:
                x.copy_(torch.randn(R, C, generator=gen, device="cuda"))
            step()                       # eager once: kernels loaded, launch shapes cached
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            step()
        replays = 5
        for i in range(replays):
            with torch.cuda.stream(s):
                for x in xs:
                    x.copy_(torch.randn(R, C, generator=gen, device="cuda"))
                graph.replay()
            torch.cuda.synchronize()
            want_rs = oracle.reduce_scatter("bf16", "avg", [host(x) for x in xs])
            want_ag = oracle.all_gather_one(want_rs, [1] * P, m * 2)
            for q in range(P):
                assert_same(host(rs[q]), want_rs[q], f"replay {i} RS rank {q}")
                assert_same(host(ag[q]), want_ag, f"replay {i} AG rank {q}")
        assert dt.dt_group_check(g) == dt.DT_OK
        # 2 barriers eager + 2 per replay, all executed on the device
        assert np.array_equal(dt.dt_debug_read_window(g), oracle.expected_window(P, 2 + 2 * replays))


def test_bucket_allreduce_graph_replays_its_cached_plan(dt):
    P, counts, cap = 3, [1000, 70_001, 7, 32_768, 5], 64 << 10
    gen = torch.Generator(device="cuda").manual_seed(12)
    grads = [[torch.empty(c, dtype=torch.bfloat16, device="cuda") for _ in range(P)] for c in counts]
    table = dt.pointer_table(grads)
    s = torch.cuda.Stream()

    def refill():
        for row in grads:
            for t in row:
                t.copy_(torch.randn(t.numel(), generator=gen, device="cuda") * 1e-3)

    with group(P) as g:
        with torch.cuda.stream(s):
            refill()
            dt.dt_bucket_allreduce(g, table, counts, "bf16", "avg", cap, s)   # builds the plan
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            dt.dt_bucket_allreduce(g, table, counts, "bf16", "avg", cap, s)   # reuses it
        for i in range(3):
            with torch.cuda.stream(s):
                refill()
            torch.cuda.synchronize()
            ref = [[host(t).copy() for t in row] for row in grads]
            with torch.cuda.stream(s):
                graph.replay()
            torch.cuda.synchronize()
            oracle.bucket_allreduce("bf16", "avg", ref)
            for t in range(len(counts)):
                for p in range(P):
                    assert_same(host(grads[t][p]), ref[t][p], f"replay {i} tensor {t} rank {p}")
        assert dt.dt_group_check(g) == dt.DT_OK
        _, nb = oracle.bucket_plan(counts, 2, cap)
        assert np.array_equal(dt.dt_debug_read_window(g), oracle.expected_window(P, 4 * (nb - 1)))


def test_captured_bucket_plan_survives_other_plans(dt):
    # A graph holds the device address of the plan it was captured with, so
    # that plan's slot is pinned: later bucket calls with other arguments use
    # other slots (new ones when needed) and the graph still replays correctly.
    P, cap = 2, 32 << 10
    gen = torch.Generator(device="cuda").manual_seed(13)

    def make(counts):
        return [[torch.empty(c, dtype=torch.float32, device="cuda") for _ in range(P)] for c in counts]

    def refill(grads):
        for row in grads:
            for t in row:
                t.copy_(torch.randn(t.numel(), generator=gen, device="cuda"))

    A, B, C = make([5000, 17, 9000]), make([300, 12000]), make([64, 64, 64, 70000])
    s = torch.cuda.Stream()
    with group(P) as g:
        with torch.cuda.stream(s):
            dt.dt_bucket_allreduce(g, A, [5000, 17, 9000], "f32", "sum", cap, s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            dt.dt_bucket_allreduce(g, A, [5000, 17, 9000], "f32", "sum", cap, s)
        for grads, counts in ((B, [300, 12000]), (C, [64, 64, 64, 70000]), (B, [300, 12000])):
            with torch.cuda.stream(s):
                refill(grads)
                dt.dt_bucket_allreduce(g, grads, counts, "f32", "sum", cap, s)
            torch.cuda.synchronize()
        with torch.cuda.stream(s):
            refill(A)
        torch.cuda.synchronize()
        ref = [[host(t).copy() for t in row] for row in A]
        with torch.cuda.stream(s):
            graph.replay()
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
    oracle.bucket_allreduce("f32", "sum", ref)
    for t in range(3):
        for p in range(P):
            assert_same(host(A[t][p]), ref[t][p], f"tensor {t} rank {p}")


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")   # the refused call captured nothing
def test_bucket_capture_without_a_cached_plan_is_refused(dt):
    P = 2
    grads = [[torch.ones(1000, device="cuda") for _ in range(P)]]
    s = torch.cuda.Stream()
    with group(P) as g:
        graph = torch.cuda.CUDAGraph()
        with pytest.raises(dt.DtError) as e:
            with torch.cuda.graph(graph, stream=s):
                dt.dt_bucket_allreduce(g, grads, [1000], "f32", "sum", 0, s)
        assert e.value.status == dt.DT_ERR_UNSUPPORTED
        torch.cuda.synchronize()
        # the group and the context are still usable
        dt.dt_bucket_allreduce(g, grads, [1000], "f32", "sum")
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
        assert float(grads[0][1][999]) == 2.0
