"""The allocation-free bucket all-reduce gives the group-based one's results.

dt_bucket_allreduce_static is for callers that cannot let a library allocate
device memory: applications whose own pool owns all device memory (a
library's cudaMalloc would escape their accounting and can fail once the pool
has taken the device) and code on a latency-critical path that must not stall
other streams (cudaMalloc and cudaFree can synchronise the whole device).
It keeps its tables in one fixed device array inside the library instead of a
group's scratch.  These tests call it through the C ABI and compare its output
with dt_bucket_allreduce's, bit for bit (the tolerance of every parity test
here), on two calls in a row with different tables, so the second call also
shows that the array's leftover contents do not leak into a result.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

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
    return t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.view(torch.int32).numpy()


def test_static_bucket_allreduce_matches_group_version_two_calls(dt):
    calls = [
        # (P, dtype, op, counts, cap): the second call has a smaller table
        (8, "bf16", "avg", [1000, 70_001, 0, 7, 32_768, 200_003, 3], 256 << 10),
        (3, "f32", "sum", [5, 40_000, 1], 64 << 10),
    ]
    for i, (P, dtype, op, counts, cap) in enumerate(calls):
        a = _grads(counts, P, dtype, 100 + i)
        b = [[x.clone() for x in row] for row in a]
        torch.cuda.synchronize()
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
    assert dt.dt_launch_count() == n0
    torch.cuda.synchronize()
    assert torch.count_nonzero(buf).item() == 0


def test_static_bucket_allreduce_full_workload(dt):
    # The 200-gradient, 8-rank bf16 workload (7 buckets of up to 25 MiB): its
    # tables (about 200 KB with one-pass bucket slices) fit the fixed array,
    # and the result equals the group-based call's, bit for bit.
    from same_device_collective_gb300 import workloads as wl
    w = wl.bucket_grads(device="cuda")
    counts = w.meta["counts"]
    a = w.inputs
    b = [[x.clone() for x in row] for row in a]
    torch.cuda.synchronize()
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
