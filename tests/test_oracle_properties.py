"""Property tests of the oracle (CPU, hypothesis): randomly drawn rank counts,
sizes and values against invariants and library routines that do not go
through the oracle's own arithmetic.

- ReduceScatter then AllGather equals AllReduce (every dtype and op).
- A 2-rank fp32 sum is one IEEE single-precision add (numpy float32).
- MAX/MIN over finite values equal numpy's maximum/minimum reduction when no
  +0/-0 tie occurs.
- AllToAll applied twice is the identity; AllToAll equals numpy's chunk
  transpose.
- The uneven AllGather equals numpy.concatenate in rank order.
- The bucket all-reduce equals the per-tensor AllReduce whatever the tensors'
  sizes.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

SETTINGS = settings(max_examples=60, deadline=None)
DTYPE_OPS = [("f32", "sum"), ("f32", "avg"), ("f32", "max"), ("f32", "min"),
             ("bf16", "sum"), ("bf16", "avg"), ("bf16", "max"), ("bf16", "min"),
             ("i32", "sum"), ("i32", "max"), ("i32", "min"), ("bf16", "sum_stepwise")]


def draw_inputs(rng: np.random.Generator, dtype: str, P: int, n: int) -> list:
    if dtype == "i32":
        return [rng.integers(-2 ** 31, 2 ** 31, n, dtype=np.int64).astype(np.int32) for _ in range(P)]
    x = [(rng.standard_normal(n) * 10.0 ** rng.integers(-3, 4)).astype(np.float32) for _ in range(P)]
    return x if dtype == "f32" else [oracle.f32_to_bf16(v) for v in x]


@SETTINGS
@given(st.integers(1, 8), st.integers(1, 40), st.sampled_from(DTYPE_OPS), st.integers(0, 2 ** 32 - 1))
def test_reduce_scatter_then_all_gather_is_allreduce(P, m, dtype_op, seed):
    dtype, op = dtype_op
    xs = draw_inputs(np.random.default_rng(seed), dtype, P, P * m)
    rs = oracle.reduce_scatter(dtype, op, xs)
    ag = oracle.all_gather(rs)
    ar = oracle.allreduce(dtype, op, xs)
    for q in range(P):
        assert np.array_equal(ag[q], ar[q].view(np.uint8))


@SETTINGS
@given(st.integers(1, 300), st.integers(0, 2 ** 32 - 1))
def test_two_rank_fp32_sum_is_one_ieee_add(n, seed):
    rng = np.random.default_rng(seed)
    a = (rng.standard_normal(n) * 10.0 ** rng.integers(-30, 30)).astype(np.float32)
    b = (rng.standard_normal(n) * 10.0 ** rng.integers(-30, 30)).astype(np.float32)
    got = oracle.allreduce("f32", "sum", [a, b])[0]
    assert np.array_equal(got.view(np.uint32), (a + b).view(np.uint32))


@SETTINGS
@given(st.integers(1, 10), st.integers(1, 200), st.sampled_from(["f32", "bf16", "i32"]),
       st.sampled_from(["max", "min"]), st.integers(0, 2 ** 32 - 1))
def test_max_min_equal_numpy_without_signed_zero_ties(P, n, dtype, op, seed):
    xs = draw_inputs(np.random.default_rng(seed), dtype, P, n)
    wide = np.stack([oracle.bf16_to_f32(x) if dtype == "bf16" else x for x in xs])
    hypothesis.assume(not np.any(wide == 0))               # no +0 / -0 ties
    got = oracle.allreduce(dtype, op, xs)[0]
    got = oracle.bf16_to_f32(got) if dtype == "bf16" else got
    want = wide.max(0) if op == "max" else wide.min(0)
    assert np.array_equal(got, want.astype(got.dtype))


@SETTINGS
@given(st.integers(1, 9), st.integers(1, 64), st.integers(0, 2 ** 32 - 1))
def test_all_to_all_is_a_chunk_transpose_and_its_own_inverse(P, c, seed):
    rng = np.random.default_rng(seed)
    xs = [rng.integers(0, 256, P * c, dtype=np.uint8) for _ in range(P)]
    out = oracle.all_to_all(xs)
    chunks = np.stack(xs).reshape(P, P, c)                  # [source i, chunk j, byte]
    for j in range(P):
        assert np.array_equal(out[j], chunks[:, j, :].reshape(-1))
    back = oracle.all_to_all(out)
    for i in range(P):
        assert np.array_equal(back[i], xs[i])


@SETTINGS
@given(st.lists(st.integers(0, 12), min_size=1, max_size=9), st.integers(1, 40),
       st.integers(0, 2 ** 32 - 1))
def test_uneven_all_gather_is_concatenation(rows, row_bytes, seed):
    rng = np.random.default_rng(seed)
    xs = [rng.integers(0, 256, r * row_bytes, dtype=np.uint8) for r in rows]
    want = np.concatenate(xs) if sum(rows) else np.zeros(0, np.uint8)
    for out in oracle.all_gather(xs, rows, row_bytes):
        assert np.array_equal(out, want)


@SETTINGS
@given(st.integers(1, 6), st.lists(st.integers(0, 300), min_size=1, max_size=8),
       st.sampled_from([("bf16", "avg"), ("bf16", "sum"), ("f32", "avg"), ("f32", "sum")]),
       st.integers(0, 2 ** 32 - 1))
def test_bucket_allreduce_is_per_tensor_allreduce(P, counts, dtype_op, seed):
    dtype, op = dtype_op
    rng = np.random.default_rng(seed)
    grads = [draw_inputs(rng, dtype, P, c) for c in counts]
    want = [oracle.allreduce(dtype, op, g) for g in grads]
    work = [[x.copy() for x in g] for g in grads]
    oracle.bucket_allreduce(dtype, op, work)
    for t in range(len(counts)):
        for p in range(P):
            assert np.array_equal(work[t][p].view(np.uint8), want[t][p].view(np.uint8))
