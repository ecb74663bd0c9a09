"""Pins of the oracle's SUM / AVG / SUM_STEPWISE at the narrowing edges.

The inputs (tests/edge_values.py) are built to reach overflow to +-Inf, the
subnormal range, Inf and NaN operands, signed zeros and exact rounding ties.
The model they are checked against is independent of the oracle: every add
and the AVG division are done in exact rational arithmetic and rounded with
the IEEE-754 definition (nearest, ties to even, gradual underflow, overflow
to Inf) written out in integers; Inf and NaN operands follow the IEEE rules
for special values; an exact zero sum is +0 unless both operands are -0.
The ascending rank order and the single narrowing at the store come from the
same-device AllReduce of the DTorch collective-communication page (§2.3) and
the hyper-parallel page's division by the world size; SUM_STEPWISE narrows
after every add, as the page's `+=` in bf16 does.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from edge_values import BF16_PATTERNS, F32_PATTERNS, as_values, edge_ranks


def _round(q: Fraction, sig_bits: int) -> float:
    """Nearest value with `sig_bits` significant bits and the binary32
    exponent range (emin -126, so subnormals are multiples of
    2^(-126 - sig_bits + 1)); ties to even; Inf past the largest finite."""
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
    quantum = Fraction(2) ** (e - sig_bits + 1)
    m = a / quantum
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    val = fl * quantum
    if val >= Fraction(2) ** 128:
        return sign * math.inf
    return sign * float(val)        # exact: every such value is a double


def rn32(q: Fraction) -> float:
    return _round(q, 24)


def rn_bf16(q: Fraction) -> float:
    return _round(q, 8)


def _special(x: float) -> bool:
    return math.isnan(x) or math.isinf(x)


def add32(a: float, b: float) -> float:
    """IEEE binary32 addition of two binary32 values."""
    if _special(a) or _special(b):
        return a + b                       # Inf/NaN rules are those of any IEEE format
    s = Fraction(a) + Fraction(b)
    if s == 0:
        both_neg = math.copysign(1.0, a) < 0 and math.copysign(1.0, b) < 0
        return -0.0 if both_neg else 0.0
    return rn32(s)


def div32(a: float, P: int) -> float:
    if _special(a) or a == 0:
        return a / P                       # keeps NaN, Inf and the sign of zero
    return rn32(Fraction(a) / P)


def narrow_bf16(a: float) -> float:
    if _special(a) or a == 0:
        return a
    return rn_bf16(Fraction(a))


def model(dtype: str, op: str, xs: list) -> float:
    """One element: xs are the P rank values (as Python floats)."""
    acc = xs[0]
    for x in xs[1:]:
        acc = add32(acc, x)
        if op == "sum_stepwise" and dtype == "bf16":
            acc = narrow_bf16(acc)
    if op == "avg":
        acc = div32(acc, len(xs))
    return narrow_bf16(acc) if dtype == "bf16" else acc


def _floats(dtype: str, bits: np.ndarray) -> np.ndarray:
    f = (bits.astype(np.uint32) << 16).view(np.float32) if dtype == "bf16" else bits.view(np.float32)
    with np.errstate(invalid="ignore"):    # signalling NaNs quieten on widening
        return f.astype(np.float64)


def _check(dtype, op, P, n, seed):
    bits, which = edge_ranks(dtype, P, n, seed)
    got = oracle.reduce(dtype, op, [as_values(dtype, b) for b in bits])
    got_f = _floats(dtype, got if dtype == "bf16" else got.view(np.uint32))
    vals = [_floats(dtype, b) for b in bits]
    for i in range(n):
        want = model(dtype, op, [float(v[i]) for v in vals])
        g = float(got_f[i])
        if math.isnan(want):
            assert math.isnan(g), (i, which[i], g)
        else:
            # bit-equal: same value and the same sign (zeros and infinities)
            assert g == want and math.copysign(1.0, g) == math.copysign(1.0, want), \
                (dtype, op, P, i, which[i], g, want)
    return got_f, which


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("op", ["sum", "avg", "sum_stepwise"])
@pytest.mark.parametrize("P", [2, 3, 4, 5, 8, 16])
def test_oracle_edge_values_equal_exact_rounding_model(dtype, op, P):
    _check(dtype, op, P, 700, 1000 * P + len(op))


def test_edge_inputs_reach_every_edge():
    """The generator does what it claims: the oracle's results on it hold
    +Inf, -Inf, NaN, nonzero subnormals and -0, for both dtypes, SUM and AVG
    (so the GPU tests that reuse these inputs cover those results)."""
    for dtype in ("bf16", "f32"):
        for op, P in (("sum", 3), ("avg", 3), ("avg", 8), ("sum", 16)):
            bits, which = edge_ranks(dtype, P, 20_000, 7)
            got = oracle.reduce(dtype, op, [as_values(dtype, b) for b in bits])
            f = _floats(dtype, got if dtype == "bf16" else got.view(np.uint32))
            assert np.any(f == np.inf) and np.any(f == -np.inf), (dtype, op, P)
            assert np.any(np.isnan(f)), (dtype, op, P)
            sub = (f != 0) & (np.abs(f) < 2.0 ** -126)
            assert np.count_nonzero(sub) > 100, (dtype, op, P)
            assert np.any((f == 0) & np.signbit(f)), (dtype, op, P)


def test_hand_tie_positions_hold_the_hand_results():
    """At every position of the 1 + 2^-8 + 2^-8 pattern the oracle's bf16
    SUM is +-0x3F81 and SUM_STEPWISE +-0x3F80 (the hand-derived values)."""
    P = 3
    bits, which = edge_ranks("bf16", P, 30_000, 11)
    pos = which == BF16_PATTERNS.index("hand_tie")
    assert np.count_nonzero(pos) > 1000
    s = oracle.reduce("bf16", "sum", bits)[pos] & 0x7FFF
    w = oracle.reduce("bf16", "sum_stepwise", bits)[pos] & 0x7FFF
    assert np.all(s == 0x3F81) and np.all(w == 0x3F80)
    # the double-rounding pattern 1 + 2^-8 + 2^-33: fp32 drops 2^-33, then
    # the bf16 tie goes to even (1.0); exact arithmetic would round up
    pos = which == BF16_PATTERNS.index("double_round")
    assert np.all(oracle.reduce("bf16", "sum", bits)[pos] & 0x7FFF == 0x3F80)


def test_f32_patterns_are_distinct_names():
    assert len(set(F32_PATTERNS)) == len(F32_PATTERNS)
    assert len(set(BF16_PATTERNS)) == len(BF16_PATTERNS)
