"""GPU parity at the narrowing edges of SUM, AVG and SUM_STEPWISE.

The inputs (tests/edge_values.py) reach sums that round past the largest
finite bf16 or fp32 value to +-Inf, sums and averages in the subnormal range
(AVG by division at P = 3 and 5, by an exact power-of-two scale at P = 2, 4,
8 and 16), +-Inf, Inf + (-Inf) and NaN operands, signed zeros, exact ties at
the fp32 add and at the bf16 store, fp32-then-bf16 double rounding, and the
hand example 1 + 2^-8 + 2^-8 (0x3F81 for SUM, 0x3F80 for SUM_STEPWISE) at
thousands of positions.  AllReduce, ReduceScatter and the bucket all-reduce
run them on the 16-byte vector path (aligned buffers, whose ragged tails take
the element path) and on the element-wise path (misaligned views), and every
result is compared with the oracle's bit for bit.  A NaN result compares by
NaN-ness only: the CPU and the GPU propagate different NaN payloads.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from edge_values import as_values, edge_ranks
from gpu_util import group, host, offset_view

pytestmark = pytest.mark.gpu

OPS = ["sum", "avg", "sum_stepwise"]


@pytest.fixture(scope="module")
def dt():
    from same_device_collective_gb300 import dt as mod
    assert torch.cuda.is_available()
    return mod


def to_device(dtype: str, bits: np.ndarray, misaligned: bool) -> torch.Tensor:
    """A device tensor holding exactly these bits; a misaligned one starts
    one element into its allocation (never 16-byte aligned)."""
    src = torch.from_numpy(bits.view(np.int16 if dtype == "bf16" else np.int32).copy())
    src = src.view(torch.bfloat16 if dtype == "bf16" else torch.float32)
    if not misaligned:
        return src.cuda()
    v = offset_view(bits.size, dtype, 1)
    v.copy_(src.cuda())
    assert v.data_ptr() % 16 != 0
    return v


def empty_out(dtype: str, n: int, misaligned: bool) -> torch.Tensor:
    if misaligned:
        return offset_view(n, dtype, 1)
    return torch.empty(n, dtype=torch.bfloat16 if dtype == "bf16" else torch.float32, device="cuda")


def bits_of(dtype: str, a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a).reshape(-1)
    return a.view(np.uint16) if dtype == "bf16" else a.view(np.uint32)


def is_nan_bits(dtype: str, b: np.ndarray) -> np.ndarray:
    if dtype == "bf16":
        return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)
    return ((b & 0x7F800000) == 0x7F800000) & ((b & 0x007FFFFF) != 0)


def assert_edge_equal(dtype: str, got: np.ndarray, want: np.ndarray, what: str):
    g, w = bits_of(dtype, got), bits_of(dtype, want)
    assert g.size == w.size, what
    ng, nw = is_nan_bits(dtype, g), is_nan_bits(dtype, w)
    if not np.array_equal(ng, nw):
        bad = np.nonzero(ng != nw)[0]
        raise AssertionError(f"{what}: NaN-ness differs at {bad.size} elements, first {bad[0]}")
    keep = ~nw
    if not np.array_equal(g[keep], w[keep]):
        idx = np.nonzero(keep)[0][g[keep] != w[keep]]
        raise AssertionError(f"{what}: {idx.size} elements differ, first {idx[0]}: "
                             f"got {int(g[idx[0]]):#x} want {int(w[idx[0]]):#x}")


@pytest.mark.parametrize("path", ["vector", "element"])
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("P", [2, 3, 4, 5, 8, 16])
def test_allreduce_edges_match_oracle(dt, P, dtype, op, path):
    n = 20_011
    bits, _ = edge_ranks(dtype, P, n, 31 * P + len(op))
    mis = path == "element"
    xs = [to_device(dtype, b, mis) for b in bits]
    outs = [empty_out(dtype, n, mis) for _ in range(P)]
    with group(P) as g:
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, outs, n, dtype, op)
        torch.cuda.synchronize()
    want = oracle.allreduce(dtype, op, [as_values(dtype, b) for b in bits])
    for q in range(P):
        assert_edge_equal(dtype, host(outs[q]), want[q], f"P={P} {dtype} {op} {path} rank {q}")


@pytest.mark.parametrize("path", ["vector", "element"])
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("P", [2, 3, 4, 5, 8, 16])
def test_reduce_scatter_edges_match_oracle(dt, P, dtype, op, path):
    mis = path == "element"
    m = 2_003 if mis else 2_000          # the vector path needs whole vectors per shard
    bits, _ = edge_ranks(dtype, P, P * m, 57 * P + len(op))
    xs = [to_device(dtype, b, mis) for b in bits]
    outs = [empty_out(dtype, m, mis) for _ in range(P)]
    with group(P) as g:
        dt.dt_reduce_scatter(g, dt.DT_ALL_RANKS, xs, outs, m, dtype, op)
        torch.cuda.synchronize()
    want = oracle.reduce_scatter(dtype, op, [as_values(dtype, b) for b in bits])
    for r in range(P):
        assert_edge_equal(dtype, host(outs[r]), want[r], f"P={P} {dtype} {op} {path} shard {r}")


@pytest.mark.parametrize("op", ["sum", "avg"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("P", [2, 3, 8, 16])
def test_bucket_allreduce_edges_match_oracle(dt, P, dtype, op):
    # several buckets under a 16 KiB cap; tensor 2 is a misaligned view on
    # every rank (element path), the rest take the vector path
    counts = [5_000, 17, 4_099, 20_000, 1, 2_048]
    misaligned = {2}
    host_bits, grads = [], []
    for t, c in enumerate(counts):
        bits, _ = edge_ranks(dtype, P, c, 1000 + 7 * t + P)
        host_bits.append(bits)
        grads.append([to_device(dtype, b, t in misaligned) for b in bits])
    ref = [[as_values(dtype, b).copy() for b in row] for row in host_bits]
    with group(P) as g:
        dt.dt_bucket_allreduce(g, grads, counts, dtype, op, bucket_cap_bytes=16 << 10)
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
    oracle.bucket_allreduce(dtype, op, ref)
    for t in range(len(counts)):
        for p in range(P):
            assert_edge_equal(dtype, host(grads[t][p]), ref[t][p],
                              f"P={P} {dtype} {op} tensor {t} rank {p}")
