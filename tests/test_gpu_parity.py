"""Parity of the CUDA collectives with the CPU oracle, element by element.

Every comparison is bit-exact: both sides combine ranks in ascending order in
fp32 (int32 wraps), divide by P once for AVG and round once to bf16, so the
results are unique.  Sizes span several 16-byte vectors, several blocks and a
ragged tail; misaligned views take the element-wise path.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from gpu_util import ELEM, TORCH_DTYPE, bytes_of, group, host, offset_view, rand_inputs

pytestmark = pytest.mark.gpu

DTYPE_OPS = [("f32", "sum"), ("f32", "avg"), ("f32", "max"), ("f32", "min"),
             ("bf16", "sum"), ("bf16", "avg"), ("bf16", "max"), ("bf16", "min"),
             ("i32", "sum"), ("i32", "max"), ("i32", "min")]


@pytest.fixture(scope="module")
def dt():
    from same_device_collective_gb300 import dt as mod
    assert torch.cuda.is_available()
    return mod


def assert_same(got: np.ndarray, want: np.ndarray, what: str):
    g, w = bytes_of(got), bytes_of(want)
    assert g.size == w.size, what
    if not np.array_equal(g, w):
        bad = np.nonzero(g != w)[0]
        raise AssertionError(f"{what}: {bad.size} bytes differ, first at byte {bad[0]}")


# --------------------------------------------------------------- AllReduce
@pytest.mark.parametrize("dtype,op", DTYPE_OPS)
@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 16])
def test_allreduce_matches_oracle(dt, dtype, op, P):
    for seed, n in enumerate([1, 7, 4095, 8192 + 3, 300_001]):
        xs = rand_inputs(P, n, dtype, seed)
        outs = [torch.empty_like(x) for x in xs]
        with group(P) as g:
            dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, outs, n, dtype, op)
            torch.cuda.synchronize()
        want = oracle.allreduce(dtype, op, [host(x) for x in xs])
        for q in range(P):
            assert_same(host(outs[q]), want[q], f"P={P} n={n} rank {q}")


@pytest.mark.parametrize("dtype,op", [("f32", "sum"), ("bf16", "avg"), ("i32", "max")])
@pytest.mark.parametrize("P", [2, 5, 8])
def test_allreduce_shared_and_in_place(dt, dtype, op, P):
    n = 50_003
    xs = rand_inputs(P, n, dtype, 11)
    want = oracle.allreduce(dtype, op, [host(x) for x in xs])
    shared = torch.empty_like(xs[0])
    with group(P) as g:
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, [shared] * P, n, dtype, op,
                        flags=dt.DT_SHARED_OUTPUT)
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, xs, n, dtype, op)       # in place
        torch.cuda.synchronize()
    assert_same(host(shared), want[0], "shared output")
    for q in range(P):
        assert_same(host(xs[q]), want[q], f"in place rank {q}")


@pytest.mark.parametrize("dtype,op", [("f32", "sum"), ("bf16", "avg"), ("bf16", "max"),
                                      ("i32", "sum")])
def test_allreduce_misaligned_views(dt, dtype, op):
    P, n = 3, 10_001
    src = rand_inputs(P, n, dtype, 5)
    xs, outs = [], []
    for r in range(P):
        v = offset_view(n, dtype, 1 + r)   # 2/4/6-byte (bf16) or 4/8/12-byte offsets
        v.copy_(src[r])
        xs.append(v)
        outs.append(offset_view(n, dtype, 3))
    with group(P) as g:
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, outs, n, dtype, op)
        torch.cuda.synchronize()
    want = oracle.allreduce(dtype, op, [host(x) for x in xs])
    for q in range(P):
        assert_same(host(outs[q]), want[q], f"misaligned rank {q}")


def test_allreduce_nan_and_signed_zero(dt):
    P, n = 3, 64
    vals = np.zeros((P, n), np.float32)
    vals[1, 0] = np.nan
    vals[0, 1], vals[1, 1] = 0.0, -0.0
    vals[0, 2], vals[1, 2] = -0.0, 0.0
    vals[2, 3] = np.inf
    vals[0, 4], vals[2, 4] = np.inf, -np.inf
    xs = [torch.from_numpy(vals[r].copy()).cuda() for r in range(P)]
    for op in ["max", "min"]:
        outs = [torch.empty_like(x) for x in xs]
        with group(P) as g:
            dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, outs, n, "f32", op)
            torch.cuda.synchronize()
        want = oracle.allreduce("f32", op, [v.copy() for v in vals])
        assert_same(host(outs[0]), want[0], op)
    outs = [torch.empty_like(x) for x in xs]
    with group(P) as g:
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, outs, n, "f32", "sum")
        torch.cuda.synchronize()
    want = oracle.allreduce("f32", "sum", [v.copy() for v in vals])[0]
    got = host(outs[0])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)                    # NaN payloads are not compared
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def _special_bits(dtype: str, P: int, n: int, seed: int) -> list:
    """Rank inputs drawn from the values MAX/MIN must treat with care: NaNs
    with distinct payloads (quiet and signalling, both signs), +0 and -0,
    subnormals of both signs, infinities, and a few normal values, so that
    ties, NaN runs and subnormal orderings occur at every rank position."""
    rng = np.random.default_rng(seed)
    if dtype == "bf16":
        pool = np.array([0x0000, 0x8000, 0x0001, 0x0002, 0x007F, 0x8001, 0x807F,
                         0x7F80, 0xFF80, 0x7FC0, 0x7FC1, 0xFFC3, 0x7F81, 0xFF85,
                         0x3F80, 0xBF80, 0x4000, 0x0080, 0x8080], np.uint16)
    else:
        pool = np.array([0x00000000, 0x80000000, 0x00000001, 0x00000002, 0x007FFFFF,
                         0x80000001, 0x807FFFFF, 0x7F800000, 0xFF800000, 0x7FC00000,
                         0x7FC00001, 0xFFC00003, 0x7F800001, 0xFF800005, 0x3F800000,
                         0xBF800000, 0x40000000, 0x00800000, 0x80800000], np.uint32)
    return [pool[rng.integers(0, pool.size, n)] for _ in range(P)]


def _device_from_bits(bits: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(bits.view(np.float32).copy()).cuda()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("op", ["max", "min"])
@pytest.mark.parametrize("P", [2, 3, 8, 12, 16])
def test_max_min_special_values_bit_exact(dt, dtype, op, P):
    # every bit compared, NaN payloads included: the result is the chosen
    # rank's element, unchanged (AllReduce, then ReduceScatter of P shards)
    m = 4099                                   # vector positions plus a ragged tail
    bits = _special_bits(dtype, P, P * m, 40 + P)
    xs = [_device_from_bits(b, dtype) for b in bits]
    n = P * m
    outs = [torch.empty_like(x) for x in xs]
    shards = [torch.empty(m, dtype=TORCH_DTYPE[dtype], device="cuda") for _ in range(P)]
    with group(P) as g:
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, outs, n, dtype, op)
        dt.dt_reduce_scatter(g, dt.DT_ALL_RANKS, xs, shards, m, dtype, op)
        torch.cuda.synchronize()
    view = np.uint16 if dtype == "bf16" else np.float32
    want = oracle.allreduce(dtype, op, [b.view(view).copy() for b in bits])
    for q in range(P):
        assert_same(host(outs[q]), want[q], f"allreduce rank {q}")
    want = oracle.reduce_scatter(dtype, op, [b.view(view).copy() for b in bits])
    for r in range(P):
        assert_same(host(shards[r]), want[r], f"reduce_scatter rank {r}")


@pytest.mark.parametrize("dtype", ["bf16", "f32", "i32"])
@pytest.mark.parametrize("P", [2, 3, 8, 16])
def test_sum_stepwise_matches_oracle(dt, dtype, P):
    # the page's literal `result += tensor`: bf16 rounds after every rank
    for seed, n in enumerate([7, 4096 * P + 5]):
        xs = rand_inputs(P, n, dtype, 500 + seed)
        outs = [torch.empty_like(x) for x in xs]
        m = n // P
        rs = [torch.empty(m, dtype=TORCH_DTYPE[dtype], device="cuda") for _ in range(P)]
        with group(P) as g:
            dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, outs, n, dtype, "sum_stepwise")
            if m:
                dt.dt_reduce_scatter(g, dt.DT_ALL_RANKS, xs, rs, m, dtype, "sum_stepwise")
            torch.cuda.synchronize()
        hx = [host(x) for x in xs]
        want = oracle.allreduce(dtype, "sum_stepwise", hx)
        for q in range(P):
            assert_same(host(outs[q]), want[q], f"AR n={n} rank {q}")
        if m:
            want = oracle.reduce_scatter(dtype, "sum_stepwise", [h[:m * P] for h in hx])
            for r in range(P):
                assert_same(host(rs[r]), want[r], f"RS m={m} rank {r}")


# ----------------------------------------------------------- ReduceScatter
@pytest.mark.parametrize("dtype,op", DTYPE_OPS)
@pytest.mark.parametrize("P", [2, 3, 4, 8, 16])
def test_reduce_scatter_matches_oracle(dt, dtype, op, P):
    for seed, m in enumerate([1, 5, 1000, 4096, 65_537]):
        xs = rand_inputs(P, P * m, dtype, 100 + seed)
        outs = [torch.empty(m, dtype=TORCH_DTYPE[dtype], device="cuda") for _ in range(P)]
        with group(P) as g:
            dt.dt_reduce_scatter(g, dt.DT_ALL_RANKS, xs, outs, m, dtype, op)
            torch.cuda.synchronize()
        want = oracle.reduce_scatter(dtype, op, [host(x) for x in xs])
        for r in range(P):
            assert_same(host(outs[r]), want[r], f"P={P} m={m} rank {r}")


def test_reduce_scatter_misaligned(dt):
    P, m = 4, 3001
    src = rand_inputs(P, P * m, "bf16", 7)
    xs = []
    for r in range(P):
        v = offset_view(P * m, "bf16", 1)
        v.copy_(src[r])
        xs.append(v)
    outs = [offset_view(m, "bf16", 3) for _ in range(P)]
    with group(P) as g:
        dt.dt_reduce_scatter(g, dt.DT_ALL_RANKS, xs, outs, m, "bf16", "avg")
        torch.cuda.synchronize()
    want = oracle.reduce_scatter("bf16", "avg", [host(x) for x in xs])
    for r in range(P):
        assert_same(host(outs[r]), want[r], f"rank {r}")


# --------------------------------------------------------------- AllGather
@pytest.mark.parametrize("P", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("row_bytes", [16, 12, 16384])
def test_all_gather_equal_and_uneven(dt, P, row_bytes):
    rng = np.random.default_rng(P * 1000 + row_bytes)
    for uneven in (False, True):
        rows = [int(v) for v in rng.integers(0, 40, P)] if uneven else [17] * P
        xs = [torch.from_numpy(rng.integers(0, 256, rows[r] * row_bytes, dtype=np.uint8)).cuda()
              for r in range(P)]
        total = sum(rows) * row_bytes
        for shared in (False, True):
            if shared:
                o = torch.full((total,), 0xAB, dtype=torch.uint8, device="cuda")
                outs = [o] * P
            else:
                outs = [torch.full((total,), 0xAB, dtype=torch.uint8, device="cuda")
                        for _ in range(P)]
            with group(P) as g:
                dt.dt_all_gather(g, dt.DT_ALL_RANKS, xs, outs, rows if uneven else None,
                                 rows[0], row_bytes,
                                 flags=dt.DT_SHARED_OUTPUT if shared else 0)
                torch.cuda.synchronize()
            want = oracle.all_gather([host(x) for x in xs], rows, row_bytes)
            for q in range(1 if shared else P):
                assert_same(host(outs[q]), want[q], f"rows={rows} shared={shared} rank {q}")


def test_all_gather_misaligned(dt):
    P, row_bytes = 3, 10
    rows = [5, 0, 9]
    xs = []
    for r in range(P):
        base = torch.randint(0, 256, (rows[r] * row_bytes + 7,), dtype=torch.uint8, device="cuda")
        xs.append(base[3:3 + rows[r] * row_bytes])
    outs = [torch.zeros(sum(rows) * row_bytes + 5, dtype=torch.uint8, device="cuda")[5:]
            for _ in range(P)]
    with group(P) as g:
        dt.dt_all_gather(g, dt.DT_ALL_RANKS, xs, outs, rows, 0, row_bytes)
        torch.cuda.synchronize()
    want = oracle.all_gather([host(x) for x in xs], rows, row_bytes)
    for q in range(P):
        assert_same(host(outs[q]), want[q], f"rank {q}")


# ---------------------------------------------------------------- AllToAll
@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("chunk_bytes", [16, 48, 1000, 65_536 + 16])
def test_all_to_all_matches_oracle(dt, P, chunk_bytes):
    rng = np.random.default_rng(P * 7 + chunk_bytes)
    xs = [torch.from_numpy(rng.integers(0, 256, P * chunk_bytes, dtype=np.uint8)).cuda()
          for _ in range(P)]
    outs = [torch.empty_like(x) for x in xs]
    back = [torch.empty_like(x) for x in xs]
    with group(P) as g:
        dt.dt_all_to_all(g, dt.DT_ALL_RANKS, xs, outs, chunk_bytes)
        dt.dt_all_to_all(g, dt.DT_ALL_RANKS, outs, back, chunk_bytes)
        torch.cuda.synchronize()
    want = oracle.all_to_all([host(x) for x in xs])
    for j in range(P):
        assert_same(host(outs[j]), want[j], f"rank {j}")
        assert_same(host(back[j]), host(xs[j]), f"twice rank {j}")


# ------------------------------------------------------ RS then AG == AR
@pytest.mark.parametrize("dtype,op", [("bf16", "avg"), ("f32", "sum"), ("i32", "min")])
def test_reduce_scatter_then_all_gather_equals_allreduce(dt, dtype, op):
    P, m = 4, 12_288
    xs = rand_inputs(P, P * m, dtype, 3)
    rs = [torch.empty(m, dtype=TORCH_DTYPE[dtype], device="cuda") for _ in range(P)]
    ag = [torch.empty(P * m, dtype=TORCH_DTYPE[dtype], device="cuda") for _ in range(P)]
    ar = [torch.empty(P * m, dtype=TORCH_DTYPE[dtype], device="cuda") for _ in range(P)]
    with group(P) as g:
        dt.dt_reduce_scatter(g, dt.DT_ALL_RANKS, xs, rs, m, dtype, op)
        dt.dt_all_gather(g, dt.DT_ALL_RANKS, rs, ag, None, 1, m * ELEM[dtype])
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, ar, P * m, dtype, op)
        torch.cuda.synchronize()
    for q in range(P):
        assert_same(host(ag[q]), host(ar[q]), f"rank {q}")


# ------------------------------------------------------------ bucket + barrier
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("op", ["avg", "sum"])
@pytest.mark.parametrize("P", [1, 2, 3, 8, 16])
def test_bucket_allreduce_matches_oracle(dt, dtype, op, P):
    rng = np.random.default_rng(P + 31)
    counts = [0, 1, 7, 1000, 40_000, 70_001, 5, 32_768, 3]
    for cap in (1, 4096, 200_000, 25 << 20):
        grads = [[torch.from_numpy(rng.standard_normal(c).astype(np.float32) * 1e-3)
                  .to(TORCH_DTYPE[dtype]).cuda() for _ in range(P)] for c in counts]
        ref = [[host(x).copy() for x in row] for row in grads]
        with group(P) as g:
            dt.dt_bucket_allreduce(g, grads, counts, dtype, op, bucket_cap_bytes=cap)
            torch.cuda.synchronize()
            win = dt.dt_debug_read_window(g)
            assert dt.dt_group_check(g) == dt.DT_OK
        oracle.bucket_allreduce(dtype, op, ref)
        for t in range(len(counts)):
            for p in range(P):
                assert_same(host(grads[t][p]), ref[t][p], f"cap={cap} tensor {t} rank {p}")
        _, nb = oracle.bucket_plan(counts, ELEM[dtype], cap)
        assert np.array_equal(win, oracle.expected_window(P, nb - 1)), f"cap={cap}"


def test_bucket_plan_reuse_across_calls(dt):
    # Two gradient sets used in turn: each call either reuses a cached plan
    # (same gradients, counts, dtype, op and cap) or rebuilds a slot.
    P = 4
    rng = np.random.default_rng(77)
    sets = {}
    for name, counts in (("A", [100, 40_000, 7]), ("B", [3000, 5, 70_000, 1])):
        grads = [[torch.from_numpy(rng.standard_normal(c).astype(np.float32) * 1e-3)
                  .to(torch.bfloat16).cuda() for _ in range(P)] for c in counts]
        sets[name] = (counts, grads, [[host(x).copy() for x in row] for row in grads])
    with group(P) as g:
        for i, name in enumerate(["A", "B", "A", "B", "A", "A"]):
            counts, grads, ref = sets[name]
            # alternate the nested-list and the prepared-table argument forms
            arg = grads if i % 2 == 0 else dt.pointer_table(grads)
            dt.dt_bucket_allreduce(g, arg, counts, "bf16", "sum", bucket_cap_bytes=64 << 10)
            oracle.bucket_allreduce("bf16", "sum", ref)
            torch.cuda.synchronize()
            for t in range(len(counts)):
                for p in range(P):
                    assert_same(host(grads[t][p]), ref[t][p], f"{name} tensor {t} rank {p}")
        assert dt.dt_group_check(g) == dt.DT_OK


def test_bucket_plan_matches_oracle_plan(dt):
    from same_device_collective_gb300 import workloads
    counts = workloads.bucket_counts()
    for cap in (1, 1 << 20, workloads.BUCKET_CAP_BYTES, 1 << 40):
        assert dt.dt_bucket_plan(counts, 2, cap) == oracle.bucket_plan(counts, 2, cap)


def test_bucket_misaligned_tensor(dt):
    P, n = 3, 1001
    grads = [[offset_view(n, "bf16", 1 + p) for p in range(P)]]
    for p in range(P):
        grads[0][p].copy_(torch.randn(n).to(torch.bfloat16))
    ref = [[host(x).copy() for x in grads[0]]]
    with group(P) as g:
        dt.dt_bucket_allreduce(g, grads, [n], "bf16", "avg")
        torch.cuda.synchronize()
    oracle.bucket_allreduce("bf16", "avg", ref)
    for p in range(P):
        assert_same(host(grads[0][p]), ref[0][p], f"rank {p}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("P", [2, 3, 8])
def test_bucket_slices_at_tensor_ends(dt, dtype, P):
    # Every block works on one slice of one tensor: slices of the bucket's
    # slice length (one pass of the block's threads: 2048 bf16 or 1024 fp32
    # elements for these sizes) cut at every tensor's end.  Counts around
    # multiples of that length, empty and one-element tensors, and two
    # tensors whose ranks are not 16-byte aligned (element path over several
    # slices) between aligned ones, in one bucket and in many.
    rng = np.random.default_rng(P * 7 + len(dtype))
    L = 2048 if dtype == "bf16" else 1024
    counts = [L, L + 1, L - 1, 1, 0, 2 * L + 7, 3 * L - 1, 8, 9, 3 * L, 5 * L + 3, L // 2]
    misaligned = {3, 6}
    for cap in (1, 3 * L * ELEM[dtype], 25 << 20):
        values = [[torch.from_numpy(rng.standard_normal(c).astype(np.float32)).to(TORCH_DTYPE[dtype])
                   for _ in range(P)] for c in counts]
        ref = [[host(v).copy() for v in row] for row in values]
        oracle.bucket_allreduce(dtype, "avg", ref)
        for entry in ("group", "static"):
            grads = []
            for t, c in enumerate(counts):
                row = []
                for p in range(P):
                    if t in misaligned:
                        x = offset_view(c, dtype, 1 + p)
                        x.copy_(values[t][p].cuda())
                    else:
                        x = values[t][p].cuda()
                    row.append(x)
                grads.append(row)
            if entry == "group":
                with group(P) as g:
                    dt.dt_bucket_allreduce(g, grads, counts, dtype, "avg", bucket_cap_bytes=cap)
                    torch.cuda.synchronize()
                    assert dt.dt_group_check(g) == dt.DT_OK
            else:
                dt.dt_bucket_allreduce_static(P, grads, counts, dtype, "avg", cap)
                torch.cuda.synchronize()
            for t in range(len(counts)):
                for p in range(P):
                    assert_same(host(grads[t][p]), ref[t][p], f"{entry} cap={cap} tensor {t} rank {p}")


@pytest.mark.parametrize("P", [1, 2, 3, 8, 16])
def test_barrier_window_matches_oracle(dt, P):
    with group(P) as g:
        for G in (1, 2, 7):
            while dt.dt_group_generation(g) < G:
                dt.dt_barrier(g)
            win = dt.dt_debug_read_window(g)
            sim, early = oracle.barrier_sim(P, G)
            assert early == 0
            assert np.array_equal(win, sim), f"P={P} G={G}"
        assert dt.dt_group_check(g) == dt.DT_OK


def test_barrier_golden_from_page(dt):
    from test_oracle_pins import read_golden
    meta, rows = read_golden("barrier_signal_rows.txt")
    P, G = int(meta["N"]), int(meta["G"])
    with group(P) as g:
        for _ in range(G):
            dt.dt_barrier(g)
        win = dt.dt_debug_read_window(g)
        for r in range(P):
            assert list(win[r]) == rows[r]
        assert dt.dt_group_check(g) == dt.DT_OK


@pytest.mark.parametrize("P,nbytes", [(2, 4096), (2, 1000), (16, 65_536), (5, 3)])
def test_ring_after_barrier(dt, P, nbytes):
    from test_oracle_pins import read_golden
    xs = [torch.full((nbytes,), r + 1, dtype=torch.uint8, device="cuda") for r in range(P)]
    stage = [torch.zeros(nbytes, dtype=torch.uint8, device="cuda") for _ in range(P)]
    outs = [torch.zeros(nbytes, dtype=torch.uint8, device="cuda") for _ in range(P)]
    with group(P) as g:
        for _ in range(3):
            for s in stage:
                s.zero_()
            dt.dt_debug_ring_after_barrier(g, xs, stage, outs, nbytes)
            torch.cuda.synchronize()
            for r in range(P):
                assert torch.all(outs[r] == (r + 1) % P + 1), f"rank {r}"
        assert dt.dt_group_check(g) == dt.DT_OK
    if P == 2:
        meta, rows = read_golden("ring_after_barrier.txt")
        assert [int(host(outs[r])[0]) - 1 for r in range(P)] == [rows[r] for r in range(P)]


# ------------------------------------------------------ failure detection
def test_barrier_timeout_is_reported_and_reset_recovers(dt):
    P = 4
    with group(P) as g:
        dt.dt_barrier(g)
        dt.dt_debug_barrier_expect(g, extra=5, timeout_ms=20)   # a threshold nobody reaches
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_ERR_TIMEOUT
        code, rank, peer, gen = dt.dt_group_error_detail(g)
        assert code == dt.DT_ERR_TIMEOUT and 0 <= rank < P and 0 <= peer < P and peer != rank
        assert gen == 2
        with pytest.raises(dt.DtError) as e:
            dt.dt_barrier(g)
        assert e.value.status in (dt.DT_ERR_TIMEOUT, dt.DT_ERR_POISONED)
        x = torch.ones(16, device="cuda")
        with pytest.raises(dt.DtError):
            dt.dt_allreduce(g, dt.DT_ALL_RANKS, [x] * P, [torch.empty_like(x) for _ in range(P)],
                            16, "f32", "sum")
        dt.dt_group_reset(g)
        assert dt.dt_group_check(g) == dt.DT_OK
        dt.dt_barrier(g)
        win = dt.dt_debug_read_window(g)
        assert np.array_equal(win, oracle.expected_window(P, 1))


# ------------------------------------------------------------ arguments
def test_invalid_arguments_are_rejected_without_launch(dt):
    P = 3
    x = [torch.ones(64, device="cuda") for _ in range(P)]
    o = [torch.empty(64, device="cuda") for _ in range(P)]
    with group(P) as g:
        n0 = dt.dt_launch_count()
        cases = [
            lambda: dt.dt_allreduce(g, dt.DT_ALL_RANKS, x, o, 64, "i32", "avg"),
            lambda: dt.dt_allreduce(g, 7, x, o, 64, "f32", "sum"),
            lambda: dt.dt_allreduce(g, dt.DT_ALL_RANKS, x, [o[0], o[0], o[1]], 64, "f32", "sum"),
            lambda: dt.dt_allreduce(g, dt.DT_ALL_RANKS, x, [x[1], o[1], o[2]], 64, "f32", "sum"),
            lambda: dt.dt_allreduce(g, dt.DT_ALL_RANKS, x, o, 64, "f32", "sum", flags=0x4),
            lambda: dt.dt_allreduce(g, dt.DT_ALL_RANKS, x, o, 64, "f32", "sum",
                                    flags=dt.DT_SHARED_OUTPUT),
            lambda: dt.dt_reduce_scatter(g, dt.DT_ALL_RANKS, x, [x[0], o[1], o[2]], 16, "f32", "sum"),
            lambda: dt.dt_all_to_all(g, dt.DT_ALL_RANKS, x, [x[0], o[1], o[2]], 64),
            lambda: dt.dt_bucket_allreduce(g, [[x[0], x[1], x[0]]], [64], "f32", "avg"),
            lambda: dt.dt_bucket_allreduce(g, [x], [64], "i32", "sum"),
            lambda: dt.dt_bucket_allreduce(g, [x], [64], "f32", "max"),
            lambda: dt.dt_allreduce(g, dt.DT_ALL_RANKS, [x[0], 0, x[2]], o, 64, "f32", "sum"),
        ]
        for i, c in enumerate(cases):
            with pytest.raises(dt.DtError):
                c()
        assert dt.dt_launch_count() == n0
        # zero-size calls succeed and launch nothing
        dt.dt_allreduce(g, dt.DT_ALL_RANKS, x, o, 0, "f32", "sum")
        dt.dt_all_to_all(g, dt.DT_ALL_RANKS, x, o, 0)
        dt.dt_reduce_scatter(g, dt.DT_ALL_RANKS, x, o, 0, "f32", "sum")
        dt.dt_all_gather(g, dt.DT_ALL_RANKS, x, o, [0, 0, 0], 0, 4)
        for t in o:
            t.fill_(-7.25)               # canary: nothing below may write
        vec = [torch.full((16,), -7.25, device="cuda") for _ in range(P * P)]
        dt.dt_bucket_allreduce(g, [o, x], [0, 0], "f32", "avg")
        dt.dt_replicate_to_shard(g, dt.DT_ALL_RANKS, x, o, None, 0, 16)
        dt.dt_all_gather_into_vec(g, dt.DT_ALL_RANKS, x, vec, None, 0, 16)
        dt.dt_all_to_all_2d(g, dt.DT_ALL_RANKS, x, o, 0, 12, 4, 0, 1)
        dt.dt_all_to_all_2d(g, dt.DT_ALL_RANKS, x, o, 6, 0, 4, 1, 0)
        assert dt.dt_launch_count() == n0
        torch.cuda.synchronize()
        assert all(bool((t == -7.25).all()) for t in o + vec)
        assert dt.dt_group_check(g) == dt.DT_OK


# --------------------------------------------------- every rank count 1..16
@pytest.mark.parametrize("P", list(range(1, 17)))
def test_every_rank_count(dt, P):
    # Each P from 1 to 16 (the kernels are compiled for at most 2, 4, 8 and 16
    # ranks and take the first P): AllReduce and ReduceScatter with the
    # special-value MAX/MIN inputs and with sums, an AllToAll whose P^2 chunks
    # of 48 KiB + 16 B go through the bulk copy, and an uneven AllGather.
    m = 1031                                                  # ragged vector tail
    for dtype, op in [("f32", "max"), ("bf16", "min"), ("bf16", "avg"), ("i32", "sum")]:
        if op in ("max", "min"):
            bits = _special_bits(dtype, P, P * m, 500 + P)
            xs = [_device_from_bits(b, dtype) for b in bits]
        else:
            xs = rand_inputs(P, P * m, dtype, 600 + P)
        outs = [torch.empty_like(x) for x in xs]
        shards = [torch.empty(m, dtype=TORCH_DTYPE[dtype], device="cuda") for _ in range(P)]
        with group(P) as g:
            dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, outs, P * m, dtype, op)
            dt.dt_reduce_scatter(g, dt.DT_ALL_RANKS, xs, shards, m, dtype, op)
            torch.cuda.synchronize()
        hx = [host(x) for x in xs]
        want = oracle.allreduce(dtype, op, hx)
        for q in range(P):
            assert_same(host(outs[q]), want[q], f"{dtype} {op} allreduce rank {q}")
        want = oracle.reduce_scatter(dtype, op, hx)
        for r in range(P):
            assert_same(host(shards[r]), want[r], f"{dtype} {op} reduce_scatter rank {r}")

    chunk = 48 * 1024 + 16
    gen = torch.Generator(device="cuda").manual_seed(700 + P)
    xs = [torch.randint(0, 256, (P * chunk,), generator=gen, dtype=torch.uint8, device="cuda")
          for _ in range(P)]
    a2a = [torch.empty_like(x) for x in xs]
    rows = [int(v) for v in torch.randint(0, 300, (P,), generator=torch.Generator().manual_seed(P))]
    row_bytes = 4096
    shard = [torch.randint(0, 256, (c * row_bytes,), generator=gen, dtype=torch.uint8, device="cuda")
             for c in rows]
    ag = [torch.empty(sum(rows) * row_bytes, dtype=torch.uint8, device="cuda") for _ in range(P)]
    with group(P) as g:
        dt.dt_all_to_all(g, dt.DT_ALL_RANKS, xs, a2a, chunk)
        dt.dt_all_gather(g, dt.DT_ALL_RANKS, shard, ag, rows, 0, row_bytes)
        torch.cuda.synchronize()
        assert dt.dt_group_check(g) == dt.DT_OK
    want = oracle.all_to_all([host(x) for x in xs])
    for j in range(P):
        assert_same(host(a2a[j]), want[j], f"all_to_all rank {j}")
    want = oracle.all_gather([host(s) for s in shard], rows, row_bytes)
    for q in range(P):
        assert_same(host(ag[q]), want[q], f"all_gather rank {q}")
