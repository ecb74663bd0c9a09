"""ctypes front end of the CPU oracle (``dt_oracle.c``) plus the step model of
the notify/wait barrier.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  Nothing here imports the CUDA library
and the CUDA library imports nothing from here.

Arrays are numpy arrays: fp32 as ``float32``, bf16 as its raw bits in
``uint16``, int32 as ``int32``.  dtype names are ``"f32"``, ``"bf16"``,
``"i32"``; op names ``"sum"``, ``"avg"``, ``"max"``, ``"min"``.

Parity status of each function (what pins it, in ``tests/test_oracle_pins.py``):
  reduce / allreduce   closed forms (all-ones, r+1, 2^r), hand-derived order
                       example, P=2 equals torch.add, error bound against the
                       exact rational sum, MAX/MIN equal torch.amax/amin,
                       int32 wrap, AVG identities.                     pinned
  f32_to_bf16          equals torch's float->bfloat16 on boundary patterns
                       and on random bit patterns.                      pinned
  reduce_scatter       shard-indexed closed form; equals the AllReduce
                       restricted to shard r; RS then AG equals AR.     pinned
  all_gather           equals torch.cat; uneven with equal rows equals the
                       equal case; row-offset closed form.              pinned
  all_to_all           applied twice is the identity; ownership-encoded
                       closed form.                                     pinned
  bucket_plan          hand-computed plans; partition/cap invariants.   pinned
  bucket_allreduce     equals per-tensor AllReduce for any cap.         pinned
  barrier_sim          window after g barriers reads g off the diagonal and
                       0 on it (the pages' [1,...,0,...,1] at g=1); no rank
                       released before all arrived.                     pinned
  barrier_step_model   the pages' edge-case table reproduced.          pinned
  replicate_to_shard   equals torch.chunk(x, P)[r]; gathering the shards
                       gives the tensor back.                           pinned
  all_gather_into_vec  each entry equals the source shard; concatenated
                       it is all_gather's output.                       pinned
  all_to_all_2d        equals torch.cat of torch.chunk for all four
                       (src, dest) pairs; (0,0) equals all_to_all; the
                       (s,d) then (d,s) round trip is the identity.     pinned
  sum_stepwise         hand example (1 + 2^-8 + 2^-8 stays 1.0); equals a
                       sequential torch bf16 `acc = acc + x`; P=2 and fp32
                       equal SUM.                                       pinned
"""
from __future__ import annotations

import ctypes
import itertools
from typing import Iterable, Sequence

import numpy as np

from . import build_oracle

DTYPES = {"f32": 0, "bf16": 1, "i32": 2}
OPS = {"sum": 0, "avg": 1, "max": 2, "min": 3, "sum_stepwise": 4}
NP_DTYPE = {"f32": np.float32, "bf16": np.uint16, "i32": np.int32}
STATUS = {0: "ok", 1: "invalid", 2: "unsupported"}

_lib = None


class OracleError(RuntimeError):
    pass


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = build_oracle.build()
        L = ctypes.CDLL(path)
        vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        vpp = ctypes.POINTER(ctypes.c_void_p)
        szp = ctypes.POINTER(ctypes.c_size_t)
        L.orc_reduce.argtypes = [i, i, i, vpp, sz, sz, vp]
        L.orc_allreduce.argtypes = [i, i, i, vpp, vpp, sz]
        L.orc_reduce_scatter.argtypes = [i, i, i, vpp, vpp, sz]
        L.orc_all_gather.argtypes = [i, vpp, vpp, szp, sz]
        L.orc_all_to_all.argtypes = [i, vpp, vpp, sz]
        L.orc_all_gather_one.argtypes = [i, vpp, vp, szp, sz]
        L.orc_replicate_to_shard.argtypes = [i, vpp, vpp, ctypes.POINTER(ctypes.c_int), sz, sz]
        L.orc_all_gather_into_vec.argtypes = [i, vpp, vpp, szp, sz]
        L.orc_all_to_all_2d.argtypes = [i, vpp, vpp, sz, sz, sz, i, i]
        L.orc_bucket_plan.argtypes = [szp, sz, sz, sz, szp, szp]
        L.orc_bucket_allreduce.argtypes = [i, i, i, vpp, szp, sz]
        L.orc_barrier_sim.argtypes = [i, i, ctypes.POINTER(ctypes.c_int32),
                                      ctypes.POINTER(ctypes.c_int32)]
        L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        L.orc_f32_to_bf16.restype = ctypes.c_uint16
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f32.restype = ctypes.c_float
        L.orc_f32_to_bf16_array.argtypes = [vp, vp, sz]
        for name in ("orc_reduce", "orc_allreduce", "orc_reduce_scatter", "orc_all_gather",
                     "orc_all_gather_one", "orc_replicate_to_shard", "orc_all_gather_into_vec",
                     "orc_all_to_all_2d",
                     "orc_all_to_all", "orc_bucket_plan", "orc_bucket_allreduce",
                     "orc_barrier_sim"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(st: int, what: str) -> None:
    if st != 0:
        raise OracleError(f"{what}: {STATUS.get(st, st)}")


def _ptrs(arrays: Sequence[np.ndarray]):
    arr = (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])
    return arr


def _contig(arrays: Iterable[np.ndarray], dtype=None) -> list:
    out = []
    for a in arrays:
        a = np.ascontiguousarray(a if dtype is None else a.view(dtype))
        out.append(a)
    return out


# ------------------------------------------------------------------ bf16
def f32_to_bf16(x) -> np.ndarray:
    """Round-to-nearest-even narrowing, array in, uint16 bits out."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f32_to_bf16_array(x.ctypes.data, out.ctypes.data, x.size)
    return out


def bf16_to_f32(h) -> np.ndarray:
    h = np.asarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------ collectives
def reduce(dtype: str, op: str, inputs: Sequence[np.ndarray], offset: int = 0,
           n: int | None = None) -> np.ndarray:
    """out[i] = narrow(scale(in_0[off+i] (+) ... (+) in_{P-1}[off+i]))."""
    ins = _contig([a.reshape(-1) for a in inputs], NP_DTYPE[dtype])
    if n is None:
        n = ins[0].size - offset
    out = np.empty(n, dtype=NP_DTYPE[dtype])
    _check(lib().orc_reduce(DTYPES[dtype], OPS[op], len(ins), _ptrs(ins), offset, n,
                            out.ctypes.data), "reduce")
    return out


def allreduce(dtype: str, op: str, inputs: Sequence[np.ndarray]) -> list:
    ins = _contig([a.reshape(-1) for a in inputs], NP_DTYPE[dtype])
    n = ins[0].size
    outs = [np.empty(n, dtype=NP_DTYPE[dtype]) for _ in ins]
    _check(lib().orc_allreduce(DTYPES[dtype], OPS[op], len(ins), _ptrs(ins), _ptrs(outs), n),
           "allreduce")
    return outs


def reduce_scatter(dtype: str, op: str, inputs: Sequence[np.ndarray]) -> list:
    ins = _contig([a.reshape(-1) for a in inputs], NP_DTYPE[dtype])
    P = len(ins)
    if ins[0].size % P:
        raise OracleError("reduce_scatter: input size not a multiple of P")
    m = ins[0].size // P
    outs = [np.empty(m, dtype=NP_DTYPE[dtype]) for _ in ins]
    _check(lib().orc_reduce_scatter(DTYPES[dtype], OPS[op], P, _ptrs(ins), _ptrs(outs), m),
           "reduce_scatter")
    return outs


def all_gather(inputs: Sequence[np.ndarray], rows: Sequence[int] | None = None,
               row_bytes: int | None = None) -> list:
    """Byte-level gather: inputs are per-rank arrays (any dtype); every rank
    gets the concatenation along dim 0 in rank order.  Returns uint8 arrays."""
    ins = [np.ascontiguousarray(a).reshape(-1).view(np.uint8) for a in inputs]
    P = len(ins)
    if rows is None:
        rows = [1] * P
        row_bytes = ins[0].size
    rows_c = (ctypes.c_size_t * P)(*rows)
    total = sum(rows) * row_bytes
    outs = [np.empty(total, dtype=np.uint8) for _ in range(P)]
    _check(lib().orc_all_gather(P, _ptrs(ins), _ptrs(outs), rows_c, row_bytes), "all_gather")
    return outs


def all_gather_one(inputs: Sequence[np.ndarray], rows: Sequence[int], row_bytes: int) -> np.ndarray:
    """The single concatenation that every rank receives (uint8)."""
    ins = [np.ascontiguousarray(a).reshape(-1).view(np.uint8) for a in inputs]
    P = len(ins)
    rows_c = (ctypes.c_size_t * P)(*rows)
    out = np.empty(sum(rows) * row_bytes, dtype=np.uint8)
    _check(lib().orc_all_gather_one(P, _ptrs(ins), out.ctypes.data, rows_c, row_bytes),
           "all_gather_one")
    return out


def replicate_to_shard(inputs: Sequence[np.ndarray], rows: int, row_bytes: int,
                       shard_idx: Sequence[int] | None = None) -> list:
    """Rank r keeps row block shard_idx[r] (default r) of its whole tensor."""
    ins = [np.ascontiguousarray(a).reshape(-1).view(np.uint8) for a in inputs]
    P = len(ins)
    if rows % P:
        raise OracleError("replicate_to_shard: rows not a multiple of P")
    outs = [np.empty(rows // P * row_bytes, dtype=np.uint8) for _ in range(P)]
    sidx = None if shard_idx is None else (ctypes.c_int * P)(*shard_idx)
    _check(lib().orc_replicate_to_shard(P, _ptrs(ins), _ptrs(outs), sidx, rows, row_bytes),
           "replicate_to_shard")
    return outs


def all_gather_into_vec(inputs: Sequence[np.ndarray], rows: Sequence[int], row_bytes: int) -> list:
    """out[q * P + r]: rank r's shard as held by rank q (uint8)."""
    ins = [np.ascontiguousarray(a).reshape(-1).view(np.uint8) for a in inputs]
    P = len(ins)
    outs = [np.empty(rows[r] * row_bytes, dtype=np.uint8) for _ in range(P) for r in range(P)]
    rows_c = (ctypes.c_size_t * P)(*rows)
    _check(lib().orc_all_gather_into_vec(P, _ptrs(ins), _ptrs(outs), rows_c, row_bytes),
           "all_gather_into_vec")
    return outs


def all_to_all_2d(inputs: Sequence[np.ndarray], src_dim: int, dest_dim: int) -> list:
    """S(src_dim) -> S(dest_dim) on 2-D arrays; returns 2-D arrays of the input dtype."""
    ins = [np.ascontiguousarray(a) for a in inputs]
    P = len(ins)
    R, C = ins[0].shape
    es = ins[0].dtype.itemsize
    h = R // P if dest_dim == 0 else R
    w = C // P if dest_dim == 1 else C
    shape = (P * h, w) if src_dim == 0 else (h, P * w)
    outs = [np.empty(shape, dtype=ins[0].dtype) for _ in range(P)]
    _check(lib().orc_all_to_all_2d(P, _ptrs(ins), _ptrs(outs), R, C, es, src_dim, dest_dim),
           "all_to_all_2d")
    return outs


def all_to_all(inputs: Sequence[np.ndarray]) -> list:
    """Byte-level all-to-all along dim 0: input i is P equal chunks."""
    ins = [np.ascontiguousarray(a).reshape(-1).view(np.uint8) for a in inputs]
    P = len(ins)
    if ins[0].size % P:
        raise OracleError("all_to_all: input size not a multiple of P")
    c = ins[0].size // P
    outs = [np.empty(ins[0].size, dtype=np.uint8) for _ in range(P)]
    _check(lib().orc_all_to_all(P, _ptrs(ins), _ptrs(outs), c), "all_to_all")
    return outs


def bucket_plan(counts: Sequence[int], elem_bytes: int, cap_bytes: int):
    T = len(counts)
    c = (ctypes.c_size_t * max(T, 1))(*counts)
    b = (ctypes.c_size_t * max(T, 1))()
    nb = ctypes.c_size_t()
    _check(lib().orc_bucket_plan(c, T, elem_bytes, cap_bytes, b, ctypes.byref(nb)),
           "bucket_plan")
    return [int(b[t]) for t in range(T)], int(nb.value)


def bucket_allreduce(dtype: str, op: str, grads: Sequence[Sequence[np.ndarray]]) -> None:
    """grads[t][p]: rank p's gradient t (contiguous, modified in place)."""
    T = len(grads)
    P = len(grads[0]) if T else 1
    flat = []
    counts = []
    for t in range(T):
        for p in range(P):
            g = grads[t][p]
            if not g.flags.c_contiguous or g.dtype != NP_DTYPE[dtype]:
                raise OracleError("bucket_allreduce: grads must be contiguous arrays of dtype")
            flat.append(g)
        counts.append(grads[t][0].size)
    cts = (ctypes.c_size_t * max(T, 1))(*counts)
    _check(lib().orc_bucket_allreduce(DTYPES[dtype], OPS[op], P, _ptrs(flat) if flat else None,
                                      cts, T), "bucket_allreduce")


def barrier_sim(P: int, generations: int):
    """Run the notify/wait barrier `generations` times with P host threads.
    Returns (window [P, P] int32, number of ranks released early)."""
    win = np.zeros((P, P), dtype=np.int32)
    early = ctypes.c_int32()
    _check(lib().orc_barrier_sim(P, generations,
                                 win.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                 ctypes.byref(early)), "barrier_sim")
    return win, int(early.value)


def expected_window(P: int, generations: int) -> np.ndarray:
    """Closed form of the window after `generations` barriers: each rank's
    row holds one count per peer (every peer notified it once per barrier)
    and 0 on its own column (a rank never notifies itself)."""
    w = np.full((P, P), generations, dtype=np.int32)
    np.fill_diagonal(w, 0)
    return w


# ------------------------------------------------------- barrier step model
class BarrierModel:
    """Explicit-interleaving model of the notify/wait barrier on P ranks.

    Each rank runs, for g = 1..G, its notify steps (one per peer) and then its
    wait steps (one per source); a schedule says which rank takes its next
    step.  A wait step whose condition fails does not advance.  The knobs
    reproduce the variants that the barrier page's edge-case table warns
    about:
      notify_op  "add" (AtomicAdd) or "set" (write `value`, overwrite)
      cmp        "ge" or "eq"
      layout     "row": rank r writes row r of the peer's window (one writer
                 per cell); "shared": every rank writes cell 0
      generation True: the g-th barrier waits for (count per barrier) * g;
                 False: every barrier waits for the first barrier's count
      skip_self  False: a rank also notifies itself
      wait_row   "src": rank r waits on row s of its own window (the row
                 that peer s writes); "self": it waits on its own row r,
                 which no peer writes (a mismatched notify/wait row)
    """

    def __init__(self, P: int, G: int = 1, notify_op: str = "add", cmp: str = "ge",
                 layout: str = "row", generation: bool = True, skip_self: bool = True,
                 wait_row: str = "src"):
        self.P, self.G = P, G
        self.notify_op, self.cmp, self.layout = notify_op, cmp, layout
        self.generation, self.skip_self = generation, skip_self
        self.wait_row = wait_row
        self.win = [[0] * P for _ in range(P)]
        self.arrived = [0] * (G + 1)
        self.early = []          # (rank, g): released before all ranks arrived
        self.done = [False] * P
        self.programs = [self._program(r) for r in range(P)]
        self.pending = [next(p) for p in self.programs]

    def _cell(self, owner: int, writer: int):
        return (owner, writer) if self.layout == "row" else (owner, 0)

    def _threshold(self, g: int) -> int:
        per_barrier = 1 if self.layout == "row" else self.P - 1
        if self.notify_op == "set":
            return 1
        return per_barrier * (g if self.generation else 1)

    def _program(self, r: int):
        P = self.P
        for g in range(1, self.G + 1):
            yield ("arrive", g)
            for q in range(P):
                if q == r and self.skip_self:
                    continue
                yield ("notify", q, g)
            srcs = [s for s in range(P) if s != r] if self.layout == "row" else [0]
            for s in srcs:
                yield ("wait", s, g)
            yield ("pass", g)
        yield ("end",)

    def _satisfied(self, r: int, s: int, g: int) -> bool:
        row = s if self.wait_row == "src" else r
        v = self.win[r][row] if self.layout == "row" else self.win[r][0]
        t = self._threshold(g)
        return v >= t if self.cmp == "ge" else v == t

    def step(self, r: int) -> bool:
        """Let rank r take one step; returns False if it could not advance."""
        if self.done[r]:
            return False
        ins = self.pending[r]
        kind = ins[0]
        if kind == "arrive":
            self.arrived[ins[1]] += 1
        elif kind == "notify":
            q = ins[1]
            o, c = self._cell(q, r)
            self.win[o][c] = self.win[o][c] + 1 if self.notify_op == "add" else 1
        elif kind == "wait":
            if not self._satisfied(r, ins[1], ins[2]):
                return False
        elif kind == "pass":
            if self.arrived[ins[1]] != self.P:
                self.early.append((r, ins[1]))
        elif kind == "end":
            self.done[r] = True
            return False
        self.pending[r] = next(self.programs[r])
        if self.pending[r][0] == "end":
            self.done[r] = True
        return True

    def run(self, schedule: Iterable[int]) -> "BarrierModel":
        for r in schedule:
            self.step(r)
        return self

    def run_to_end(self, order: Sequence[int] | None = None, max_rounds: int = 100000) -> bool:
        """Round-robin in `order` until every rank ends; False on deadlock."""
        order = list(order) if order is not None else list(range(self.P))
        for _ in range(max_rounds):
            if all(self.done):
                return True
            progressed = False
            for r in order:
                progressed |= self.step(r)
            if not progressed and not all(self.done):
                return False
        return all(self.done)


def all_schedules(P: int, length: int):
    """Every sequence of `length` rank ids (exhaustive, small P only)."""
    return itertools.product(range(P), repeat=length)
