"""Stream order of the bucket all-reduce against the work queued before it.

Every bucket kernel of a call after the first loads its first gradients
before waiting for the previous kernel, and the call's first kernel lets the
next launch begin only after its own wait.  Here each gradient is written by
a GEMM (cuBLAS) or a copy queued on the same stream immediately before the
call, with no host synchronisation in between, across many buckets and both
entry points; the results must equal the oracle's on the values the
producers write.  A bucket kernel that read a gradient before its producer
finished would return a sum of stale values.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import group, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dt():
    from same_device_collective_gb300 import dt as mod
    assert torch.cuda.is_available()
    return mod


def producers(P, T, seed):
    """Per tensor t and rank p, GEMM operands whose bf16 product is the
    gradient (T tensors of 256 x 256 = 65536 elements)."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    a = [torch.randn(256, 128, generator=g, device="cuda").bfloat16() for _ in range(P)]
    b = [torch.randn(128, 256, generator=g, device="cuda").bfloat16() * 0.01 for _ in range(T)]
    return a, b


@pytest.mark.parametrize("static", [False, True])
@pytest.mark.parametrize("P", [2, 8])
def test_bucket_call_after_gemms_on_the_same_stream(dt, static, P):
    T = 12
    a, b = producers(P, T, seed=40 + P)
    # the values the producers write (computed once, apart, for the oracle)
    ref = [[torch.matmul(a[p], b[t]) for p in range(P)] for t in range(T)]
    torch.cuda.synchronize()
    want = [[host(ref[t][p]).copy() for p in range(P)] for t in range(T)]
    oracle.bucket_allreduce("bf16", "avg", want)

    grads = [[torch.full((256, 256), 3.0, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
             for _ in range(T)]
    table = dt.pointer_table(grads)
    counts = np.full(T, 256 * 256, dtype=np.uint64)
    cap = 2 * 256 * 256 * 2            # two tensors per bucket: 6 buckets, 5 barriers
    stream = torch.cuda.current_stream()
    with group(P) as grp:
        for rep in range(3):
            torch.cuda.synchronize()
            torch.cuda._sleep(200_000)      # keep the producers queued behind a busy GPU
            for t in range(T):
                for p in range(P):
                    torch.matmul(a[p], b[t], out=grads[t][p])
            if static:
                dt.dt_bucket_allreduce_static(P, table, counts, "bf16", "avg", cap, stream.cuda_stream)
            else:
                dt.dt_bucket_allreduce(grp, table, counts, "bf16", "avg", cap, stream.cuda_stream)
            torch.cuda.synchronize()
            for t in range(T):
                for p in range(P):
                    got = host(grads[t][p])
                    assert np.array_equal(got, want[t][p].reshape(-1)), (rep, t, p)
        assert dt.dt_group_check(grp) == dt.DT_OK


def test_bucket_call_after_copies_on_the_same_stream(dt):
    # plain copy kernels as producers, one bucket per tensor
    P, T = 4, 16
    gen = torch.Generator(device="cuda").manual_seed(9)
    src = [[(torch.rand(70001, generator=gen, device="cuda") - 0.5).bfloat16() for _ in range(P)]
           for _ in range(T)]
    want = [[host(x).copy() for x in row] for row in src]
    oracle.bucket_allreduce("bf16", "sum", want)
    grads = [[torch.zeros(70001, dtype=torch.bfloat16, device="cuda") for _ in range(P)] for _ in range(T)]
    table = dt.pointer_table(grads)
    counts = np.full(T, 70001, dtype=np.uint64)
    with group(P) as grp:
        torch.cuda.synchronize()
        torch.cuda._sleep(200_000)
        for t in range(T):
            for p in range(P):
                grads[t][p].copy_(src[t][p])
        dt.dt_bucket_allreduce(grp, table, counts, "bf16", "sum", 1)
        torch.cuda.synchronize()
        for t in range(T):
            for p in range(P):
                assert np.array_equal(host(grads[t][p]), want[t][p]), (t, p)
