"""Pins of the CPU oracle against facts fixed outside it.

Each test ties one oracle function to something other than its own formula:
a value the pages print, a closed form, an invariant, a library routine that
the special case reduces to, the exact rational result within its error
bound, or a hand-derived value.  The last block plants plausible mistakes
(by feeding the oracle permuted arguments, on the CPU) and checks that a pin
catches each one.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(20261202)


# ----------------------------------------------------------- helpers
def f32(x):
    return np.asarray(x, dtype=np.float32)


def bits32(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


def torch_bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x_f32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def rn_f32(q: Fraction) -> float:
    """Round an exact rational to the nearest binary32, ties to even (the
    IEEE-754 definition, done in integer arithmetic)."""
    if q == 0:
        return 0.0
    sign = -1.0 if q < 0 else 1.0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    quantum = Fraction(2) ** (e - 23)
    m = a / quantum
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    val = fl * quantum
    if val >= Fraction(2) ** 128:
        return sign * float("inf")
    return sign * float(val)


def read_golden(name):
    rows = {}
    meta = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("rank"):
                head, vals = line.split(":")
                rows[int(head.split()[1])] = [int(v) for v in vals.split()]
            elif line.startswith("y "):
                _, r, _, _, s = line.split()
                rows[int(r)] = int(s)
            else:
                k, v = line.split(None, 1)
                meta[k] = v
    return meta, rows


# ------------------------------------------------------- bf16 narrowing
def test_bf16_narrow_matches_torch_on_boundary_patterns():
    uppers = [0x0000, 0x0001, 0x007F, 0x0080, 0x0081, 0x3F80, 0x3F81, 0x3FFF, 0x4780,
              0x7F7E, 0x7F7F, 0x7F80, 0x8000, 0x8001, 0x8080, 0xBF80, 0xFF7F, 0xFF80]
    lowers = [0x0000, 0x0001, 0x4000, 0x7FFF, 0x8000, 0x8001, 0xC000, 0xFFFF]
    pats = np.array([(u << 16) | l for u in uppers for l in lowers], dtype=np.uint32)
    x = pats.view(np.float32)
    ours = oracle.f32_to_bf16(x)
    ref = torch_bf16_bits(x)
    finite = ~np.isnan(x)          # NaN payloads are a convention, checked below
    assert np.array_equal(ours[finite], ref[finite])
    assert np.all(np.isnan(oracle.bf16_to_f32(ours[~finite])))


def test_bf16_narrow_matches_torch_on_random_bits():
    pats = rng.integers(0, 2 ** 32, size=1 << 18, dtype=np.uint64).astype(np.uint32)
    x = pats.view(np.float32)
    finite = np.isfinite(x)
    ours = oracle.f32_to_bf16(x)
    ref = torch_bf16_bits(x)
    assert np.array_equal(ours[finite], ref[finite])
    # NaNs stay NaNs with their sign
    nan = np.isnan(x)
    back = oracle.bf16_to_f32(ours[nan])
    assert np.all(np.isnan(back))
    assert np.array_equal(np.signbit(back), np.signbit(x[nan]))


def test_bf16_narrow_hand_values():
    # bf16 has 8 significant bits: around 1.0 its ulp is 2^-7, half an ulp 2^-8.
    cases = {
        1.0 + 2.0 ** -8: 0x3F80,          # exact tie, 0x3F80 is even: stays
        1.0 + 3 * 2.0 ** -8: 0x3F82,      # tie between 0x3F81 and 0x3F82: even
        1.0 + 2.0 ** -8 + 2.0 ** -20: 0x3F81,   # just above the tie: up
        3.4028234663852886e38: 0x7F80,    # largest binary32 rounds past bf16 max: inf
        -0.0: 0x8000,
        2.0 ** -133: 0x0001,              # smallest bf16 subnormal, exact
    }
    for v, want in cases.items():
        assert int(oracle.f32_to_bf16(f32([v]))[0]) == want, v


# ------------------------------------------------------ reduce: closed forms
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("P", [1, 2, 3, 5, 8, 16])
def test_allreduce_closed_forms(dtype, P):
    n = 37
    def mk(v):
        if dtype == "i32":
            return np.full(n, v, dtype=np.int32)
        if dtype == "bf16":
            return oracle.f32_to_bf16(np.full(n, v, dtype=np.float32))
        return np.full(n, v, dtype=np.float32)

    def val(a):
        return oracle.bf16_to_f32(a) if dtype == "bf16" else a

    # all ones -> P
    outs = oracle.allreduce(dtype, "sum", [mk(1) for _ in range(P)])
    for o in outs:
        assert np.all(val(o) == P)
    # rank r holds r + 1 -> P (P + 1) / 2   (exact: at most 136 < 2^8)
    outs = oracle.allreduce(dtype, "sum", [mk(r + 1) for r in range(P)])
    for o in outs:
        assert np.all(val(o) == P * (P + 1) // 2)
    # rank r holds 2^r -> 2^P - 1 (binary32 and int32 exact; bf16 rounds once)
    outs = oracle.allreduce(dtype, "sum", [mk(2 ** r) for r in range(P)])
    want = 2 ** P - 1
    if dtype == "bf16":
        want = float(torch.tensor(float(want)).to(torch.bfloat16))
    for o in outs:
        assert np.all(val(o) == want)
    # MAX / MIN select the largest / smallest rank value
    outs = oracle.allreduce(dtype, "max", [mk(r) for r in range(P)])
    assert np.all(val(outs[0]) == P - 1)
    outs = oracle.allreduce(dtype, "min", [mk(-r) for r in range(P)])
    assert np.all(val(outs[0]) == -(P - 1))
    if dtype != "i32":
        # AVG of all ones is 1, AVG of r + 1 is (P + 1) / 2 (exact for these P)
        outs = oracle.allreduce(dtype, "avg", [mk(1) for _ in range(P)])
        assert np.all(val(outs[0]) == 1)
        outs = oracle.allreduce(dtype, "avg", [mk(r + 1) for r in range(P)])
        assert np.all(val(outs[0]) == (P + 1) / 2)


def test_sum_order_is_ascending_rank_hand_example():
    # 1 + 2^-24 is exactly half an ulp above 1: ties to even give 1, twice.
    # Adding the two small terms first would give 1 + 2^-23 instead.
    ins = [f32([1.0]), f32([2.0 ** -24]), f32([2.0 ** -24])]
    out = oracle.reduce("f32", "sum", ins)
    assert out[0] == np.float32(1.0)
    rev = oracle.reduce("f32", "sum", ins[::-1])
    assert rev[0] == np.float32(1.0 + 2.0 ** -23)


def test_bf16_accumulates_in_fp32_and_rounds_once_hand_example():
    # 1 + 2^-8 + 2^-8 = 1 + 2^-7 exactly in fp32 -> bf16 0x3F81.  Rounding to
    # bf16 after every add would give 1 (each 1 + 2^-8 is a tie to even).
    ins = [oracle.f32_to_bf16(f32([v])) for v in (1.0, 2.0 ** -8, 2.0 ** -8)]
    out = oracle.reduce("bf16", "sum", ins)
    assert int(out[0]) == 0x3F81


def test_sum_stepwise_rounds_every_add_hand_example():
    # the page's `result += tensor` in bf16: 1 + 2^-8 is a tie and rounds to 1.0
    # (even), twice, so the result stays 0x3F80 where SUM gives 0x3F81
    ins = [oracle.f32_to_bf16(f32([v])) for v in (1.0, 2.0 ** -8, 2.0 ** -8)]
    assert int(oracle.reduce("bf16", "sum_stepwise", ins)[0]) == 0x3F80
    assert int(oracle.reduce("bf16", "sum", ins)[0]) == 0x3F81


@pytest.mark.parametrize("P", [2, 3, 5, 8, 16])
def test_sum_stepwise_equals_sequential_torch_bf16_adds(P):
    xs = [oracle.f32_to_bf16(rng.uniform(-1, 1, 2049).astype(np.float32)) for _ in range(P)]
    t = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) for x in xs]
    acc = t[0].clone()
    for r in range(1, P):
        acc = acc + t[r]              # torch bf16 add: exact fp32 sum, one RNE to bf16
    ref = acc.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.reduce("bf16", "sum_stepwise", xs), ref)


def test_sum_stepwise_is_sum_for_two_ranks_fp32_and_int32():
    xs = [oracle.f32_to_bf16(rng.uniform(-1, 1, 999).astype(np.float32)) for _ in range(2)]
    assert np.array_equal(oracle.reduce("bf16", "sum_stepwise", xs), oracle.reduce("bf16", "sum", xs))
    fs = [rng.uniform(-1, 1, 999).astype(np.float32) for _ in range(5)]
    assert np.array_equal(oracle.reduce("f32", "sum_stepwise", fs), oracle.reduce("f32", "sum", fs))
    ii = [rng.integers(-2 ** 31, 2 ** 31, 99, dtype=np.int64).astype(np.int32) for _ in range(5)]
    assert np.array_equal(oracle.reduce("i32", "sum_stepwise", ii), oracle.reduce("i32", "sum", ii))


def test_two_rank_fp32_sum_equals_torch_add():
    a = rng.standard_normal(4099).astype(np.float32) * 1e3
    b = rng.standard_normal(4099).astype(np.float32)
    ours = oracle.allreduce("f32", "sum", [a, b])
    ref = (torch.from_numpy(a) + torch.from_numpy(b)).numpy()
    for o in ours:
        assert np.array_equal(bits32(o), bits32(ref))


@pytest.mark.parametrize("P", [2, 3])
def test_brute_force_exact_rounding_small(P):
    """P <= 3, N <= 64: the sum equals the exact rational sum of rank 0 and
    rank 1 rounded once to binary32, then (P = 3) plus rank 2 rounded again --
    exact arithmetic plus the IEEE rounding definition, no float adds."""
    n = 64
    xs = [(rng.standard_normal(n) * 10.0 ** rng.integers(-6, 6, n)).astype(np.float32)
          for _ in range(P)]
    out = oracle.reduce("f32", "sum", xs)
    for i in range(n):
        acc = Fraction(float(xs[0][i]))
        for r in range(1, P):
            acc = Fraction(rn_f32(acc + Fraction(float(xs[r][i]))))
        assert float(out[i]) == rn_f32(acc), i


@pytest.mark.parametrize("P", [3, 4, 7, 16])
def test_sum_within_recursive_summation_bound(P):
    n = 256
    xs = [rng.uniform(-1, 1, n).astype(np.float32) for _ in range(P)]
    out = oracle.reduce("f32", "sum", xs)
    u = 2.0 ** -24
    gamma = (P - 1) * u / (1 - (P - 1) * u)
    for i in range(n):
        exact = sum(Fraction(float(x[i])) for x in xs)
        bound = gamma * sum(abs(float(x[i])) for x in xs)
        assert abs(float(out[i]) - float(exact)) <= bound * (1 + 1e-12)


@pytest.mark.parametrize("P", [2, 4, 8, 16])
def test_avg_power_of_two_is_exact_scaling(P):
    # x / 2^k and x * 2^-k are the same real number, so both round the same.
    xs = [rng.uniform(-1, 1, 1000).astype(np.float32) for _ in range(P)]
    s = oracle.reduce("f32", "sum", xs)
    a = oracle.reduce("f32", "avg", xs)
    assert np.array_equal(bits32(a), bits32(np.ldexp(s, -int(np.log2(P))).astype(np.float32)))


def test_avg_non_power_of_two_rounds_once():
    xs = [f32([1.0]), f32([2.0]), f32([4.0])]
    a = oracle.reduce("f32", "avg", xs)
    assert float(a[0]) == rn_f32(Fraction(7, 3))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("op", ["max", "min"])
def test_max_min_equal_torch_amax_amin(dtype, op):
    P, n = 5, 3001
    xs = [rng.uniform(-1, 1, n).astype(np.float32) for _ in range(P)]
    if dtype == "bf16":
        xs = [oracle.f32_to_bf16(x) for x in xs]
        t = torch.stack([torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) for x in xs])
    else:
        t = torch.stack([torch.from_numpy(x) for x in xs])
    ref = (t.amax(0) if op == "max" else t.amin(0))
    ref = ref.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else ref.numpy()
    out = oracle.reduce(dtype, op, xs)
    assert np.array_equal(out.view(np.uint8), ref.view(np.uint8))


def test_max_min_nan_and_signed_zero_hand_cases():
    nan = np.float32("nan")
    assert np.isnan(oracle.reduce("f32", "max", [f32([1.0]), f32([nan]), f32([2.0])])[0])
    assert np.isnan(oracle.reduce("f32", "max", [f32([nan]), f32([5.0])])[0])
    assert np.isnan(oracle.reduce("f32", "min", [f32([3.0]), f32([nan])])[0])
    # equal values keep the lower rank's bits: +0 vs -0
    assert bits32(oracle.reduce("f32", "max", [f32([0.0]), f32([-0.0])]))[0] == 0x00000000
    assert bits32(oracle.reduce("f32", "max", [f32([-0.0]), f32([0.0])]))[0] == 0x80000000
    assert bits32(oracle.reduce("f32", "min", [f32([0.0]), f32([-0.0])]))[0] == 0x00000000


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("op", ["max", "min"])
def test_max_min_special_values_closed_form(dtype, op):
    # Inputs from NaNs with distinct payloads, +-0, subnormals, infinities and
    # normals.  Closed form of the selection rule, element by element: if any
    # rank holds a NaN, the result is the highest such rank's element, bits
    # unchanged; otherwise it is the element of the lowest rank whose value
    # equals numpy's max (min) of the widened values.
    if dtype == "bf16":
        pool = np.array([0x0000, 0x8000, 0x0001, 0x007F, 0x8001, 0x807F, 0x7F80, 0xFF80,
                         0x7FC0, 0x7FC1, 0xFFC3, 0x7F81, 0x3F80, 0xBF80, 0x0080], np.uint16)
        widen = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        pool = np.array([0x00000000, 0x80000000, 0x00000001, 0x007FFFFF, 0x80000001,
                         0x7F800000, 0xFF800000, 0x7FC00000, 0x7FC00001, 0xFFC00003,
                         0x7F800001, 0x3F800000, 0xBF800000, 0x00800000], np.uint32)
        widen = lambda b: b.view(np.float32).astype(np.float64)
    P, n = 6, 4000
    r = np.random.default_rng(7)
    bits = np.stack([pool[r.integers(0, pool.size, n)] for _ in range(P)])
    vals = widen(bits.reshape(-1)).reshape(P, n)
    ins = [bits[p].view(np.uint16 if dtype == "bf16" else np.float32).copy() for p in range(P)]
    got = oracle.reduce(dtype, op, ins).view(bits.dtype)
    isnan = np.isnan(vals)
    last_nan = P - 1 - np.argmax(isnan[::-1], axis=0)
    clean = np.where(isnan, -np.inf if op == "max" else np.inf, vals)
    best = clean.max(0) if op == "max" else clean.min(0)
    first_best = np.argmax(clean == best, axis=0)
    pick = np.where(isnan.any(0), last_nan, first_best)
    assert np.array_equal(got, bits[pick, np.arange(n)])


def test_int32_sum_wraps_and_max_min_equal_numpy():
    big = np.array([2 ** 31 - 1], dtype=np.int32)
    one = np.array([1], dtype=np.int32)
    assert int(oracle.reduce("i32", "sum", [big, one])[0]) == -2 ** 31
    xs = [rng.integers(-2 ** 31, 2 ** 31, 999, dtype=np.int64).astype(np.int32) for _ in range(6)]
    assert np.array_equal(oracle.reduce("i32", "max", xs), np.max(np.stack(xs), 0))
    assert np.array_equal(oracle.reduce("i32", "min", xs), np.min(np.stack(xs), 0))
    wide = np.sum(np.stack(xs).astype(np.int64), 0)
    assert np.array_equal(oracle.reduce("i32", "sum", xs), wide.astype(np.uint64).astype(np.uint32)
                          .view(np.int32))


def test_unsupported_and_invalid_arguments():
    with pytest.raises(oracle.OracleError, match="unsupported"):
        oracle.reduce("i32", "avg", [np.zeros(4, np.int32)] * 2)
    with pytest.raises(oracle.OracleError, match="reduce_scatter"):
        oracle.reduce_scatter("f32", "sum", [np.zeros(5, np.float32)] * 2)


# ----------------------------------------------------- reduce-scatter
@pytest.mark.parametrize("P", [2, 3, 4, 8])
def test_reduce_scatter_shard_closed_form(P):
    m = 50
    # rank p's element k holds 1000 p + k: shard r of the sum is
    # 1000 P (P - 1) / 2 + P (r m + i), exact in fp32 at these sizes.
    xs = [(1000.0 * p + np.arange(P * m)).astype(np.float32) for p in range(P)]
    outs = oracle.reduce_scatter("f32", "sum", xs)
    for r in range(P):
        want = 1000.0 * P * (P - 1) / 2 + P * (r * m + np.arange(m))
        assert np.array_equal(outs[r], want.astype(np.float32))


@pytest.mark.parametrize("dtype,op", [("f32", "sum"), ("bf16", "avg"), ("i32", "max"),
                                      ("bf16", "min")])
def test_reduce_scatter_is_allreduce_restricted_to_shard(dtype, op):
    P, m = 4, 333
    xs = [rng.uniform(-1, 1, P * m).astype(np.float32) for _ in range(P)]
    if dtype == "bf16":
        xs = [oracle.f32_to_bf16(x) for x in xs]
    if dtype == "i32":
        xs = [(x * 2 ** 20).astype(np.int32) for x in xs]
    ar = oracle.allreduce(dtype, op, xs)[0]
    rs = oracle.reduce_scatter(dtype, op, xs)
    for r in range(P):
        assert np.array_equal(rs[r].view(np.uint8), ar[r * m:(r + 1) * m].view(np.uint8))


@pytest.mark.parametrize("dtype,op", [("f32", "sum"), ("bf16", "avg"), ("i32", "sum"),
                                      ("f32", "max")])
def test_reduce_scatter_then_all_gather_equals_allreduce(dtype, op):
    P, m = 8, 129
    xs = [rng.uniform(-1, 1, P * m).astype(np.float32) for _ in range(P)]
    if dtype == "bf16":
        xs = [oracle.f32_to_bf16(x) for x in xs]
    if dtype == "i32":
        xs = [(x * 2 ** 20).astype(np.int32) for x in xs]
    rs = oracle.reduce_scatter(dtype, op, xs)
    ag = oracle.all_gather(rs)
    ar = oracle.allreduce(dtype, op, xs)
    for q in range(P):
        assert np.array_equal(ag[q], ar[q].view(np.uint8))


# --------------------------------------------------------- all-gather
def test_all_gather_equals_torch_cat():
    P = 5
    xs = [rng.integers(0, 255, (7, 12), dtype=np.uint8) for _ in range(P)]
    outs = oracle.all_gather(xs)
    ref = torch.cat([torch.from_numpy(x) for x in xs], 0).numpy().reshape(-1)
    for o in outs:
        assert np.array_equal(o, ref)


def test_uneven_all_gather_row_offsets_closed_form():
    rows = [3, 1, 4, 1, 5]
    row_bytes = 6
    xs = [np.full(c * row_bytes, r + 1, dtype=np.uint8) for r, c in enumerate(rows)]
    outs = oracle.all_gather(xs, rows, row_bytes)
    want = np.concatenate([np.full(c * row_bytes, r + 1, np.uint8) for r, c in enumerate(rows)])
    for o in outs:
        assert np.array_equal(o, want)
    # rank 2's first row starts at row 3 + 1 = 4
    assert outs[0][4 * row_bytes] == 3


def test_all_gather_one_equals_every_rank_output():
    rows = [3, 0, 5, 2]
    xs = [rng.integers(0, 255, c * 8, dtype=np.uint8) for c in rows]
    full = oracle.all_gather(xs, rows, 8)
    one = oracle.all_gather_one(xs, rows, 8)
    ref = torch.cat([torch.from_numpy(x) for x in xs]).numpy()
    assert np.array_equal(one, ref)
    for o in full:
        assert np.array_equal(o, one)


def test_uneven_with_equal_rows_equals_equal_gather():
    P, rows, rb = 4, 3, 20
    xs = [rng.integers(0, 255, rows * rb, dtype=np.uint8) for _ in range(P)]
    a = oracle.all_gather(xs)
    b = oracle.all_gather(xs, [rows] * P, rb)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_uneven_all_gather_zero_rows():
    rows = [0, 2, 0]
    xs = [np.zeros(0, np.uint8), np.arange(8, dtype=np.uint8), np.zeros(0, np.uint8)]
    outs = oracle.all_gather(xs, rows, 4)
    for o in outs:
        assert np.array_equal(o, np.arange(8, dtype=np.uint8))


# --------------------------------------------------------- all-to-all
@pytest.mark.parametrize("P", [1, 2, 3, 8])
def test_all_to_all_ownership_closed_form(P):
    c = 5
    # rank i's chunk j holds the value i * P + j
    xs = [np.repeat(np.arange(P, dtype=np.int32) + i * P, c) for i in range(P)]
    outs = [o.view(np.int32) for o in oracle.all_to_all(xs)]
    for j in range(P):
        assert np.array_equal(outs[j], np.repeat(np.arange(P, dtype=np.int32) * P + j, c))


@pytest.mark.parametrize("P", [2, 4, 8])
def test_all_to_all_twice_is_identity(P):
    xs = [rng.integers(0, 255, P * 24, dtype=np.uint8) for _ in range(P)]
    once = oracle.all_to_all(xs)
    twice = oracle.all_to_all(once)
    for x, y in zip(xs, twice):
        assert np.array_equal(x, y)


# --------------------------------------- ReplicateToShard, IntoVec, 2-D A2A
@pytest.mark.parametrize("P", [1, 2, 4, 5])
def test_replicate_to_shard_equals_torch_chunk_and_gathers_back(P):
    rows, cols = 6 * P, 7
    x = rng.integers(0, 255, (rows, cols), dtype=np.uint8)
    outs = oracle.replicate_to_shard([x] * P, rows, cols)
    for r in range(P):
        assert np.array_equal(outs[r], torch.chunk(torch.from_numpy(x), P, 0)[r].numpy().reshape(-1))
    back = oracle.all_gather(outs)
    assert np.array_equal(back[0], x.reshape(-1))
    # an explicit shard index picks another block
    outs = oracle.replicate_to_shard([x] * P, rows, cols, shard_idx=[P - 1 - r for r in range(P)])
    assert np.array_equal(outs[0], torch.chunk(torch.from_numpy(x), P, 0)[P - 1].numpy().reshape(-1))
    if P > 1:
        with pytest.raises(oracle.OracleError):
            oracle.replicate_to_shard([x] * P, rows + 1, cols)


@pytest.mark.parametrize("P", [1, 3, 4])
def test_all_gather_into_vec_entries_and_concatenation(P):
    rows = [2 + r for r in range(P)]
    xs = [rng.integers(0, 255, rows[r] * 8, dtype=np.uint8) for r in range(P)]
    vec = oracle.all_gather_into_vec(xs, rows, 8)
    for q in range(P):
        for r in range(P):
            assert np.array_equal(vec[q * P + r], xs[r])
        assert np.array_equal(np.concatenate(vec[q * P:(q + 1) * P]),
                              oracle.all_gather(xs, rows, 8)[q])


@pytest.mark.parametrize("P", [1, 2, 4])
@pytest.mark.parametrize("src_dim,dest_dim", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_all_to_all_2d_equals_torch_chunk_cat(P, src_dim, dest_dim):
    R, C = 4 * P, 6 * P
    xs = [rng.integers(-1000, 1000, (R, C)).astype(np.int32) for _ in range(P)]
    outs = oracle.all_to_all_2d(xs, src_dim, dest_dim)
    ts = [torch.from_numpy(x) for x in xs]
    for j in range(P):
        ref = torch.cat([torch.chunk(t, P, dest_dim)[j] for t in ts], src_dim)
        assert np.array_equal(outs[j], ref.numpy())
    back = oracle.all_to_all_2d(outs, dest_dim, src_dim)
    for x, b in zip(xs, back):
        assert np.array_equal(x, b)


def test_all_to_all_2d_dim0_equals_flat_all_to_all():
    P = 4
    xs = [rng.integers(0, 255, (8, 12), dtype=np.uint8) for _ in range(P)]
    a = oracle.all_to_all_2d(xs, 0, 0)
    b = oracle.all_to_all(xs)
    for x, y in zip(a, b):
        assert np.array_equal(x.reshape(-1), y)


def test_planted_wrong_split_dim_is_caught():
    P = 2
    xs = [rng.integers(0, 255, (4, 6), dtype=np.uint8) for _ in range(P)]
    mutant = oracle.all_to_all_2d(xs, 0, 0)            # split along the wrong dim
    ts = [torch.from_numpy(x) for x in xs]
    ref = torch.cat([torch.chunk(t, P, 1)[0] for t in ts], 0).numpy()
    assert mutant[0].shape != ref.shape or not np.array_equal(mutant[0], ref)


# ----------------------------------------------------------- buckets
def test_bucket_plan_hand_cases():
    assert oracle.bucket_plan([10, 10, 10], 2, 40) == ([0, 0, 1], 2)
    assert oracle.bucket_plan([30, 5, 30], 2, 40) == ([0, 1, 2], 3)
    assert oracle.bucket_plan([5, 5, 5, 5], 2, 20) == ([0, 0, 1, 1], 2)
    assert oracle.bucket_plan([], 2, 40) == ([], 0)
    assert oracle.bucket_plan([0, 100, 1], 2, 10) == ([0, 0, 1], 2)


def test_bucket_plan_invariants_random():
    counts = [int(c) for c in rng.integers(0, 5000, 300)]
    es, cap = 2, 4096
    b, nb = oracle.bucket_plan(counts, es, cap)
    assert b[0] == 0 and b[-1] == nb - 1
    assert all(b[t + 1] - b[t] in (0, 1) for t in range(len(b) - 1))
    for k in range(nb):
        members = [t for t in range(len(b)) if b[t] == k]
        size = sum(counts[t] * es for t in members)
        nonzero = [t for t in members if counts[t] > 0]
        assert size <= cap or len(nonzero) == 1
        if k + 1 < nb:   # greedy: the next tensor did not fit
            nxt = members[-1] + 1
            assert size + counts[nxt] * es > cap


def test_bucket_allreduce_equals_per_tensor_allreduce():
    P, counts = 3, [5, 17, 1, 64]
    grads = [[oracle.f32_to_bf16(rng.standard_normal(c).astype(np.float32) * 1e-3)
              for _ in range(P)] for c in counts]
    want = [oracle.allreduce("bf16", "avg", g) for g in grads]
    oracle.bucket_allreduce("bf16", "avg", grads)
    for t in range(len(counts)):
        for p in range(P):
            assert np.array_equal(grads[t][p], want[t][p])


def test_bucket_config_plan_has_about_eight_buckets():
    from same_device_collective_gb300 import workloads
    counts = workloads.bucket_counts()
    assert len(counts) == 200 and min(counts) >= 1000 and max(counts) <= 4_000_000
    _, nb = oracle.bucket_plan(counts, 2, workloads.BUCKET_CAP_BYTES)
    total = sum(counts) * 2
    assert nb >= -(-total // workloads.BUCKET_CAP_BYTES)
    assert 4 <= nb <= 16


# ------------------------------------------------------------ barrier
def test_barrier_golden_from_page():
    meta, rows = read_golden("barrier_signal_rows.txt")
    P, G = int(meta["N"]), int(meta["G"])
    win, early = oracle.barrier_sim(P, G)
    assert early == 0
    for r in range(P):
        assert list(win[r]) == rows[r]
    assert meta["expect"] == "OK"


@pytest.mark.parametrize("P,G", [(2, 1), (3, 5), (8, 17), (16, 40)])
def test_barrier_window_after_g_generations(P, G):
    win, early = oracle.barrier_sim(P, G)
    assert early == 0
    assert np.array_equal(win, oracle.expected_window(P, G))


def test_barrier_step_model_never_releases_early_exhaustive():
    # every interleaving of 12 steps on 3 ranks, two generations, then run out
    P, G = 3, 2
    for sched in oracle.all_schedules(P, 8):
        m = oracle.BarrierModel(P, G)
        m.run(sched)
        assert m.run_to_end()
        assert m.early == []
        assert [row[:] for row in m.win] == oracle.expected_window(P, G).tolist()


def test_barrier_step_model_edge_cases_from_page():
    P = 3
    # Set/Eq on one shared cell: released as soon as the first peer arrives
    m = oracle.BarrierModel(P, 1, notify_op="set", cmp="eq", layout="shared")
    m.run([1, 1, 0, 0, 0, 0, 0])      # rank 1 arrives and notifies rank 0; rank 0 runs
    assert (0, 1) in m.early
    # AtomicAdd/Ge on the shared cell with threshold P-1 is correct
    m = oracle.BarrierModel(P, 1, notify_op="add", cmp="ge", layout="shared")
    m.run([1, 1, 0, 0, 0, 0, 0])
    assert m.early == []
    assert m.run_to_end() and m.early == []
    # reuse without a generation: the second barrier passes on stale counts
    m = oracle.BarrierModel(P, 2, generation=False)
    assert m.run_to_end([0, 1, 2]) is True
    m = oracle.BarrierModel(P, 2, generation=False)
    for _ in range(100):                   # everyone finishes barrier 1 ...
        behind = [r for r in range(P) if m.pending[r] != ("arrive", 2)]
        if not behind:
            break
        m.run(behind)
    m.run([0] * 6)                         # ... then rank 0 runs barrier 2 alone
    assert (0, 2) in m.early
    m = oracle.BarrierModel(P, 2, generation=True)
    for _ in range(100):
        behind = [r for r in range(P) if m.pending[r] != ("arrive", 2)]
        if not behind:
            break
        m.run(behind)
    m.run([0] * 6)                         # with the generation, rank 0 must wait
    assert m.early == [] and m.pending[0][0] == "wait"
    # a rank that does not skip itself leaves a count on its own column
    m = oracle.BarrierModel(P, 1, skip_self=False)
    assert m.run_to_end()
    assert all(m.win[r][r] == 1 for r in range(P))
    # a wait on the wrong row never ends
    m = oracle.BarrierModel(P, 1, wait_row="self")
    assert m.run_to_end(max_rounds=200) is False


def test_ring_golden_ordering_after_barrier_model():
    """y[r] = x[(r+1) % N] holds when the load happens after the barrier: in the
    step model, a rank that passes barrier 1 sees every rank arrived (staged)."""
    meta, rows = read_golden("ring_after_barrier.txt")
    N = int(meta["N"])
    for sched in oracle.all_schedules(N, 6):
        m = oracle.BarrierModel(N, 1)
        m.run(sched)
        m.run_to_end()
        assert m.early == []
    x = np.arange(N) * 10 + 7
    y = np.array([x[(r + 1) % N] for r in range(N)])
    assert [int(np.where(x == v)[0][0]) for v in y] == [rows[r] for r in range(N)]


# ------------------------------------------------- planted mistakes caught
def test_planted_descending_order_is_caught():
    ins = [f32([1.0]), f32([2.0 ** -24]), f32([2.0 ** -24])]
    mutant = oracle.reduce("f32", "sum", ins[::-1])      # ranks combined high to low
    assert mutant[0] != np.float32(1.0)


def test_planted_dropped_rank_is_caught():
    P = 4
    xs = [np.full(3, r + 1, np.float32) for r in range(P)]
    mutant = oracle.reduce("f32", "sum", xs[:-1])        # last rank dropped
    assert not np.all(mutant == P * (P + 1) // 2)


def test_planted_wrong_shard_is_caught():
    P, m = 4, 10
    xs = [(1000.0 * p + np.arange(P * m)).astype(np.float32) for p in range(P)]
    r = 1
    mutant = oracle.reduce("f32", "sum", xs, offset=((r + 1) % P) * m, n=m)   # shard r+1
    want = 1000.0 * P * (P - 1) / 2 + P * (r * m + np.arange(m))
    assert not np.array_equal(mutant, want.astype(np.float32))


def test_planted_transposed_all_to_all_is_caught():
    P, c = 3, 2
    xs = [np.repeat(np.arange(P, dtype=np.int32) + i * P, c) for i in range(P)]
    mutant = [x.copy() for x in xs]                     # "out_j = in_j": no exchange
    good = [o.view(np.int32) for o in oracle.all_to_all(xs)]
    assert any(not np.array_equal(a, b) for a, b in zip(mutant, good))


def test_planted_missing_avg_divide_is_caught():
    xs = [np.full(4, 1, np.float32) for _ in range(4)]
    mutant = oracle.reduce("f32", "sum", xs)           # AVG without the divide
    assert not np.all(mutant == 1)
