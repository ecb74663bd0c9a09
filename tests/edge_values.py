"""Seeded rank inputs that reach the edges of the SUM / AVG / SUM_STEPWISE
narrowing: sums that round past the largest finite value to +-Inf, sums and
averages in the subnormal range, +-Inf and NaN inputs, Inf + (-Inf), signed
zeros, exact round-to-nearest-even ties at the fp32 add and at the bf16 store,
and the double rounding of an fp32 sum that is then narrowed to bf16.

Only bit patterns are built here; nothing reduces them.  Every element index
draws one pattern, which fixes that element's value on every rank, so a long
enough array places each pattern at thousands of positions, inside 16-byte
vectors and in ragged tails alike.  Arrays hold raw bits: uint16 for bf16,
uint32 for fp32.
"""
from __future__ import annotations

import numpy as np

BF16_PATTERNS = ["overflow", "tie_to_inf", "below_inf", "subnormal", "tiny_normal", "inf",
                 "inf_minus_inf", "nan", "hand_tie", "store_tie", "double_round", "normal",
                 "signed_zero", "cancel"]
F32_PATTERNS = ["overflow", "tie_to_inf", "below_inf", "subnormal", "tiny_normal", "inf",
                "inf_minus_inf", "nan", "add_tie", "normal", "signed_zero", "cancel"]


def _bf16_bits_of(v: np.ndarray) -> np.ndarray:
    """Exact float32 -> bf16 bits for values that bf16 represents (the low
    16 bits must be zero; checked)."""
    b = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value not representable in bf16"
    return (b >> 16).astype(np.uint16)


def _pattern_bf16(name: str, P: int, k: int, rng) -> np.ndarray:
    """[P, k] bf16 bits for k positions of one pattern."""
    out = np.zeros((P, k), dtype=np.uint16)
    sign = (rng.integers(0, 2, k) << 15).astype(np.uint16)
    if name in ("overflow", "tie_to_inf", "below_inf"):
        # rank 0 the largest finite bf16 (2 - 2^-7) * 2^127; rank 1 another
        # bf16 max (the fp32 sum overflows), half a bf16 ulp of it, 2^119
        # (an exact fp32 sum on the tie, which rounds to the even Inf), or a
        # quarter ulp, 2^118 (rounds back to the max)
        second = {"overflow": 0x7F7F, "tie_to_inf": 0x7B00, "below_inf": 0x7A80}[name]
        out[0] = 0x7F7F | sign
        if P > 1:
            out[1] = second | sign
    elif name == "subnormal":
        out[:] = rng.integers(1, 0x80, (P, k)).astype(np.uint16) | \
            (rng.integers(0, 2, (P, k)) << 15).astype(np.uint16)
    elif name == "tiny_normal":
        # exponent fields 1..3: normal values below 2^-123, whose sums cancel
        # into the subnormal range and whose averages fall into it
        e = rng.integers(1, 4, (P, k)).astype(np.uint16)
        m = rng.integers(0, 0x80, (P, k)).astype(np.uint16)
        out[:] = (e << 7) | m | (rng.integers(0, 2, (P, k)) << 15).astype(np.uint16)
    elif name in ("inf", "inf_minus_inf", "nan", "normal", "cancel"):
        v = rng.standard_normal((P, k)).astype(np.float32)
        out[:] = (v.view(np.uint32) >> 16).astype(np.uint16)
        cols = np.arange(k)
        a = rng.integers(0, P, k)
        if name == "inf":
            out[a, cols] = 0x7F80 | sign
        elif name == "inf_minus_inf" and P > 1:
            b = (a + rng.integers(1, P, k)) % P
            out[a, cols] = 0x7F80
            out[b, cols] = 0xFF80
        elif name == "nan":
            # quiet and signalling payloads, both signs
            out[a, cols] = 0x7F80 | rng.integers(1, 0x80, k).astype(np.uint16) | sign
        elif name == "cancel" and P > 1:
            out[1] = out[0] ^ 0x8000          # rank 1 = -rank 0, exactly
            if P > 2:                         # much smaller values on the other ranks
                small = (rng.standard_normal((P - 2, k)) * 2.0 ** -20).astype(np.float32)
                out[2:] = (small.view(np.uint32) >> 16).astype(np.uint16)
    elif name == "hand_tie":
        # 1 + 2^-8 + 2^-8: exactly 1 + 2^-7 in fp32 (0x3F81 after the store);
        # rounding after every add gives 1 (each 1 + 2^-8 is a tie to even)
        out[0] = 0x3F80 | sign
        if P > 1:
            out[1] = 0x3B80 | sign
        if P > 2:
            out[2] = 0x3B80 | sign
    elif name == "store_tie":
        # rank 0 a random normal a = m * 2^E, rank 1 +-2^(E-8), half a bf16
        # ulp of a: the fp32 sum is exact and sits on a rounding tie (or, when
        # it lowers a power of two, on a representable value)
        e = rng.integers(40, 200, k).astype(np.uint16)
        m = rng.integers(0, 0x80, k).astype(np.uint16)
        out[0] = (e << 7) | m | sign
        if P > 1:
            out[1] = ((e - 8) << 7) | (rng.integers(0, 2, k) << 15).astype(np.uint16)
    elif name == "double_round":
        # 1 + 2^-8 + 2^-33: the fp32 add of 2^-33 rounds away (below half an
        # fp32 ulp), leaving the bf16 tie 1 + 2^-8, which rounds to 1; the
        # exact sum would round up.  Both sides must round twice, in order.
        out[0] = 0x3F80 | sign
        if P > 1:
            out[1] = 0x3B80 | sign
        if P > 2:
            out[2] = _bf16_bits_of(np.full(k, 2.0 ** -33, np.float32)) | sign
    elif name == "signed_zero":
        out[:] = (rng.integers(0, 2, (P, k)) << 15).astype(np.uint16)
        allneg = rng.integers(0, 2, k).astype(bool)
        out[:, allneg] = 0x8000               # -0 on every rank sums to -0
    else:
        raise ValueError(name)
    return out


def _pattern_f32(name: str, P: int, k: int, rng) -> np.ndarray:
    """[P, k] fp32 bits for k positions of one pattern."""
    out = np.zeros((P, k), dtype=np.uint32)
    sign = (rng.integers(0, 2, k).astype(np.uint32) << 31)
    if name in ("overflow", "tie_to_inf", "below_inf"):
        # rank 0 the largest finite fp32 (2 - 2^-23) * 2^127; rank 1 the max
        # again, half its ulp (2^103: the add is a tie and rounds to the even
        # Inf), or a quarter ulp (2^102: rounds back to the max)
        second = {"overflow": 0x7F7FFFFF, "tie_to_inf": (103 + 127) << 23,
                  "below_inf": (102 + 127) << 23}[name]
        out[0] = 0x7F7FFFFF | sign
        if P > 1:
            out[1] = np.uint32(second) | sign
    elif name == "subnormal":
        out[:] = rng.integers(1, 1 << 23, (P, k)).astype(np.uint32) | \
            (rng.integers(0, 2, (P, k)).astype(np.uint32) << 31)
    elif name == "tiny_normal":
        e = rng.integers(1, 4, (P, k)).astype(np.uint32)
        m = rng.integers(0, 1 << 23, (P, k)).astype(np.uint32)
        out[:] = (e << 23) | m | (rng.integers(0, 2, (P, k)).astype(np.uint32) << 31)
    elif name in ("inf", "inf_minus_inf", "nan", "normal", "cancel"):
        out[:] = rng.standard_normal((P, k)).astype(np.float32).view(np.uint32)
        cols = np.arange(k)
        a = rng.integers(0, P, k)
        if name == "inf":
            out[a, cols] = 0x7F800000 | sign
        elif name == "inf_minus_inf" and P > 1:
            b = (a + rng.integers(1, P, k)) % P
            out[a, cols] = 0x7F800000
            out[b, cols] = 0xFF800000
        elif name == "nan":
            out[a, cols] = 0x7F800000 | rng.integers(1, 1 << 23, k).astype(np.uint32) | sign
        elif name == "cancel" and P > 1:
            out[1] = out[0] ^ np.uint32(0x80000000)
    elif name == "add_tie":
        # rank 0 a random normal a = m * 2^E, rank 1 +-2^(E-24), half an fp32
        # ulp of a: the first add is a round-to-nearest-even tie
        e = rng.integers(40, 200, k).astype(np.uint32)
        out[0] = (e << 23) | rng.integers(0, 1 << 23, k).astype(np.uint32) | sign
        if P > 1:
            out[1] = ((e - 24) << 23) | (rng.integers(0, 2, k).astype(np.uint32) << 31)
    elif name == "signed_zero":
        out[:] = rng.integers(0, 2, (P, k)).astype(np.uint32) << 31
        allneg = rng.integers(0, 2, k).astype(bool)
        out[:, allneg] = 0x80000000
    else:
        raise ValueError(name)
    return out


def edge_ranks(dtype: str, P: int, n: int, seed: int):
    """P rank arrays of n elements (raw bits) and the pattern index of every
    element (into BF16_PATTERNS or F32_PATTERNS)."""
    rng = np.random.default_rng(seed)
    names = BF16_PATTERNS if dtype == "bf16" else F32_PATTERNS
    which = rng.integers(0, len(names), n)
    bits_t = np.uint16 if dtype == "bf16" else np.uint32
    out = np.zeros((P, n), dtype=bits_t)
    for i, name in enumerate(names):
        cols = np.nonzero(which == i)[0]
        if cols.size:
            maker = _pattern_bf16 if dtype == "bf16" else _pattern_f32
            out[:, cols] = maker(name, P, cols.size, rng)
    return [out[r].copy() for r in range(P)], which


def as_values(dtype: str, bits: np.ndarray) -> np.ndarray:
    """Raw bits in the array type the oracle takes: uint16 bf16 bits stay as
    they are, fp32 bits become float32."""
    return bits if dtype == "bf16" else bits.view(np.float32)
