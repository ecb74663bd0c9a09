"""The allocation-free bucket all-reduce gives the group-based one's results.

dt_bucket_allreduce_static is for callers that cannot let a library allocate
device memory: applications whose own pool owns all device memory (a
library's cudaMalloc would escape their accounting and can fail once the pool
has taken the device) and code on a latency-critical path that must not stall
other streams (cudaMalloc and cudaFree can synchronise the whole device).
It keeps its tables in one fixed device array inside the library instead of a
group's scratch.  These tests call it through the C ABI and compare its output
with dt_bucket_allreduce's and with the oracle's, bit for bit (the tolerance
of every parity test here), on calls in a row with different tables, so a
later call also shows that the array's leftover contents do not leak into a
result; calls queued back to back on one stream with no host wait between
them; a call that repeats the previous call's tables (reused on the device
without a copy); and a call on a capturing stream, which is refused.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dt():
    from same_device_collective_gb300 import dt as mod
    assert torch.cuda.is_available()
    return mod


def _grads(counts, P, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    return [[(torch.randn(c, generator=g) * 1e-3).to(td).cuda() for _ in range(P)]
            for c in counts]


def _host(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 \
        else t.numpy()


def _oracle_after(grads, dtype, op, times=1):
    """The oracle's result of `times` bucket all-reduces of these gradients
    (taken from the device before any call runs)."""
    ref = [[_host(x).copy() for x in row] for row in grads]
    for _ in range(times):
        oracle.bucket_allreduce(dtype, op, ref)
    return ref


def _assert_equal(grads, ref, what):
    for t in range(len(grads)):
        for p in range(len(grads[t])):
            a, b = _host(grads[t][p]), ref[t][p]
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), f"{what}: tensor {t} rank {p}"


CALLS = [
    # (P, dtype, op, counts, cap): the second call has a smaller table
    (8, "bf16", "avg", [1000, 70_001, 0, 7, 32_768, 200_003, 3], 256 << 10),
    (3, "f32", "sum", [5, 40_000, 1], 64 << 10),
]


def test_static_bucket_allreduce_matches_group_version_and_oracle_two_calls(dt):
    for i, (P, dtype, op, counts, cap) in enumerate(CALLS):
        a = _grads(counts, P, dtype, 100 + i)
        b = [[x.clone() for x in row] for row in a]
        torch.cuda.synchronize()
        ref = _oracle_after(a, dtype, op)
        dt.dt_bucket_allreduce_static(P, a, counts, dtype, op, bucket_cap_bytes=cap)
        g = dt.dt_group_create(P, torch.cuda.current_device())
        try:
            dt.dt_bucket_allreduce(g, b, counts, dtype, op, bucket_cap_bytes=cap)
            torch.cuda.synchronize()
            assert dt.dt_group_check(g) == dt.DT_OK
        finally:
            dt.dt_group_destroy(g)
        for t in range(len(counts)):
            for p in range(P):
                assert np.array_equal(_host(a[t][p]), _host(b[t][p])), f"call {i} tensor {t} rank {p}"
        _assert_equal(a, ref, f"call {i} against the oracle")


def test_static_calls_back_to_back_on_one_stream(dt):
    # Three calls queued on one stream with no host wait between them, each
    # with other tables than the one before (different ranks and dtypes, then
    # the first call's shapes on new buffers): every result equals the
    # oracle's.
    s = torch.cuda.Stream()
    sets = [_grads(counts, P, dtype, 200 + i) for i, (P, dtype, op, counts, cap) in enumerate(CALLS)]
    again = _grads(CALLS[0][3], CALLS[0][0], CALLS[0][1], 300)
    torch.cuda.synchronize()
    refs = [_oracle_after(sets[i], c[1], c[2]) for i, c in enumerate(CALLS)]
    ref_again = _oracle_after(again, CALLS[0][1], CALLS[0][2])
    order = [(sets[0], CALLS[0]), (sets[1], CALLS[1]), (again, CALLS[0])]
    with torch.cuda.stream(s):
        for grads, (P, dtype, op, counts, cap) in order:
            dt.dt_bucket_allreduce_static(P, grads, counts, dtype, op, bucket_cap_bytes=cap, stream=s)
    torch.cuda.synchronize()
    _assert_equal(sets[0], refs[0], "first call")
    _assert_equal(sets[1], refs[1], "second call")
    _assert_equal(again, ref_again, "third call (first call's shapes, new buffers)")


def test_static_call_repeating_its_tables_reuses_them(dt):
    # The same gradients twice in a row on one stream: the second call finds
    # its tables on the device already.  The result is the oracle's bucket
    # all-reduce applied twice.
    P, dtype, op, counts, cap = CALLS[0]
    a = _grads(counts, P, dtype, 400)
    torch.cuda.synchronize()
    ref = _oracle_after(a, dtype, op, times=2)
    dt.dt_bucket_allreduce_static(P, a, counts, dtype, op, bucket_cap_bytes=cap)
    dt.dt_bucket_allreduce_static(P, a, counts, dtype, op, bucket_cap_bytes=cap)
    torch.cuda.synchronize()
    _assert_equal(a, ref, "repeated call")
    # the same gradients under another cap: other buckets, other tables,
    # which must be copied (the result does not depend on the buckets)
    ref3 = _oracle_after(a, dtype, op)
    dt.dt_bucket_allreduce_static(P, a, counts, dtype, op, bucket_cap_bytes=cap // 4)
    torch.cuda.synchronize()
    _assert_equal(a, ref3, "call with another cap")


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_static_call_on_a_capturing_stream_is_refused(dt):
    # The refused call enqueues nothing; the capture stays valid: work
    # captured after it replays, and the gradients are untouched.
    P = 2
    grads = [[torch.ones(1000, device="cuda") for _ in range(P)]]
    dt.dt_bucket_allreduce_static(P, grads, [1000], "f32", "sum")   # eager: 1 + 1 = 2
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    x = torch.zeros(16, device="cuda")
    n0 = dt.dt_launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        with pytest.raises(dt.DtError) as e:
            dt.dt_bucket_allreduce_static(P, grads, [1000], "f32", "sum", stream=s)
        x.add_(1.0)
    assert e.value.status == dt.DT_ERR_UNSUPPORTED
    assert dt.dt_launch_count() == n0
    graph.replay()
    torch.cuda.synchronize()
    assert torch.all(x == 1.0)
    assert torch.all(grads[0][0] == 2.0) and torch.all(grads[0][1] == 2.0)
    # and the next eager call works
    dt.dt_bucket_allreduce_static(P, grads, [1000], "f32", "sum")
    torch.cuda.synchronize()
    assert torch.all(grads[0][0] == 4.0)


def test_static_bucket_allreduce_rejects_tables_past_the_fixed_array(dt):
    # Every pointer below is real, distinct device memory, so the check is
    # exercised without ever handing a kernel an address it may not touch.
    P = 16
    T = 8200                      # 8200 * 16 pointers * 8 B > 1 MiB of pointer table
    buf = torch.zeros(T * P * 8, dtype=torch.bfloat16, device="cuda")
    base = buf.data_ptr()
    grads = [[base + (t * P + p) * 16 for p in range(P)] for t in range(T)]
    n0 = dt.dt_launch_count()
    with pytest.raises(dt.DtError) as e:
        dt.dt_bucket_allreduce_static(P, grads, [1] * T, "bf16", "avg")
    assert e.value.status == dt.DT_ERR_TOO_LARGE
    # more buckets than the fixed launch list holds: one tensor per bucket
    T = 5000
    grads = [[base + (t * 2 + p) * 16 for p in range(2)] for t in range(T)]
    with pytest.raises(dt.DtError) as e:
        dt.dt_bucket_allreduce_static(2, grads, [1] * T, "bf16", "sum", bucket_cap_bytes=1)
    assert e.value.status == dt.DT_ERR_TOO_LARGE
    # overlapping gradients are refused before anything is enqueued
    grads = [[base, base + 64], [base + 96, base + 32]]     # tensor 1 rank 1 overlaps rank 0 of tensor 0
    with pytest.raises(dt.DtError) as e:
        dt.dt_bucket_allreduce_static(2, grads, [32, 32], "bf16", "sum")
    assert e.value.status == dt.DT_ERR_INVALID
    assert dt.dt_launch_count() == n0
    torch.cuda.synchronize()
    assert torch.count_nonzero(buf).item() == 0


def test_static_bucket_allreduce_full_workload(dt):
    # The 200-gradient, 8-rank bf16 workload (7 buckets of up to 25 MiB): its
    # tables (about 400 KB with one-pass bucket slices) fit the fixed array,
    # and the result equals the group-based call's and the oracle's, bit for
    # bit (the oracle on 20 of the 200 gradients, spread over every bucket).
    from same_device_collective_gb300 import workloads as wl
    w = wl.bucket_grads(device="cuda")
    counts = w.meta["counts"]
    a = w.inputs
    b = [[x.clone() for x in row] for row in a]
    sample = list(range(0, len(counts), 10))
    torch.cuda.synchronize()
    ref = _oracle_after([a[t] for t in sample], "bf16", "avg")
    dt.dt_bucket_allreduce_static(8, a, counts, "bf16", "avg", bucket_cap_bytes=wl.BUCKET_CAP_BYTES)
    g = dt.dt_group_create(8, torch.cuda.current_device())
    try:
        dt.dt_bucket_allreduce(g, b, counts, "bf16", "avg", bucket_cap_bytes=wl.BUCKET_CAP_BYTES)
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
    finally:
        dt.dt_group_destroy(g)
    for t in range(len(counts)):
        for p in range(8):
            assert torch.equal(a[t][p], b[t][p]), f"tensor {t} rank {p}"
    _assert_equal([a[t] for t in sample], ref, "sampled tensors against the oracle")
