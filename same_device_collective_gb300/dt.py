"""Python binding of the dt C ABI (include/dt.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does
nothing but turn Python arguments into C ones: tensors become their
``data_ptr()``, lists become pointer arrays, a stream argument of ``None``
becomes PyTorch's current stream on the group's device.  Every collective runs
in the CUDA kernels of ``libdt.so``; there is no other code path.  Importing
this module without the built library raises ``ImportError``.
"""
from __future__ import annotations

import ctypes
import inspect
import os
import re
from typing import Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdt.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "dt.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`"
        " (the collectives have no non-CUDA implementation)")

_lib = ctypes.CDLL(LIB_PATH)

DT_OK, DT_ERR_INVALID, DT_ERR_UNSUPPORTED, DT_ERR_CUDA, DT_ERR_TIMEOUT, DT_ERR_OOM, \
    DT_ERR_POISONED, DT_ERR_TOO_LARGE, DT_NOT_READY = range(9)
DT_F32, DT_BF16, DT_I32 = 0, 1, 2
DT_SUM, DT_AVG, DT_MAX, DT_MIN, DT_SUM_STEPWISE = 0, 1, 2, 3, 4
DT_MAX_RANKS = 16
DT_ALL_RANKS = -1
DT_SHARED_OUTPUT = 0x1
DT_DEFAULT_BUCKET_CAP_BYTES = 25 << 20
DT_BUILD_NVTX, DT_BUILD_TIMELINE, DT_BUILD_BOUNDS = 1, 2, 4
BOUNDS_KERNELS = {1: "reduce", 2: "reduce_shift", 3: "copy_bulk", 4: "copy_vec", 5: "copy_edge",
                  6: "copy_shift", 7: "copy_2d", 8: "bucket"}

DTYPES = {"f32": DT_F32, "bf16": DT_BF16, "i32": DT_I32}
OPS = {"sum": DT_SUM, "avg": DT_AVG, "max": DT_MAX, "min": DT_MIN,
       "sum_stepwise": DT_SUM_STEPWISE}

_vp = ctypes.c_void_p
_vpp = ctypes.POINTER(ctypes.c_void_p)
_sz = ctypes.c_size_t
_szp = ctypes.POINTER(ctypes.c_size_t)
_i = ctypes.c_int
_u = ctypes.c_uint
_u32 = ctypes.c_uint32

_SIGS = {
    "dt_group_create": ([_i, _i, ctypes.POINTER(_vp)], _i),
    "dt_group_destroy": ([_vp], _i),
    "dt_group_reset": ([_vp, _vp], _i),
    "dt_group_check": ([_vp], _i),
    "dt_group_error_detail": ([_vp, ctypes.POINTER(_i), ctypes.POINTER(_i), ctypes.POINTER(_i)], _i),
    "dt_group_size": ([_vp], _i),
    "dt_group_generation": ([_vp], ctypes.c_int64),
    "dt_group_set_timeout_ms": ([_vp, _u32], _i),
    "dt_status_string": ([_i], ctypes.c_char_p),
    "dt_launch_count": ([], ctypes.c_uint64),
    "dt_allreduce": ([_vp, _i, _vpp, _vpp, _sz, _i, _i, _u, _vp], _i),
    "dt_reduce_scatter": ([_vp, _i, _vpp, _vpp, _sz, _i, _i, _vp], _i),
    "dt_all_gather": ([_vp, _i, _vpp, _vpp, _szp, _sz, _sz, _u, _vp], _i),
    "dt_all_to_all": ([_vp, _i, _vpp, _vpp, _sz, _vp], _i),
    "dt_bucket_allreduce": ([_vp, _vpp, _szp, _sz, _i, _i, _sz, _vp], _i),
    "dt_bucket_plan": ([_szp, _sz, _sz, _sz, _szp, _szp], _i),
    "dt_bucket_allreduce_static": ([_i, _vpp, _szp, _sz, _i, _i, _sz, _vp], _i),
    "dt_barrier": ([_vp, _i, _vp], _i),
    "dt_replicate_to_shard": ([_vp, _i, _vpp, _vpp, ctypes.POINTER(_i), _sz, _sz, _vp], _i),
    "dt_all_gather_into_vec": ([_vp, _i, _vpp, _vpp, _szp, _sz, _sz, _vp], _i),
    "dt_all_to_all_2d": ([_vp, _i, _vpp, _vpp, _sz, _sz, _sz, _i, _i, _vp], _i),
    "dt_async_begin": ([_vp, _vp, ctypes.POINTER(_vp)], _i),
    "dt_async_end": ([_vp, ctypes.POINTER(_vp)], _i),
    "dt_work_wait": ([_vp, _vp], _i),
    "dt_work_query": ([_vp], _i),
    "dt_work_free": ([_vp], _i),
    "dt_debug_read_window": ([_vp, ctypes.POINTER(ctypes.c_int32), _vp], _i),
    "dt_debug_ring_after_barrier": ([_vp, _vpp, _vpp, _vpp, _sz, _vp], _i),
    "dt_debug_barrier_expect": ([_vp, _i, _u32, _vp], _i),
    "dt_timeline_start": ([_sz], _i),
    "dt_timeline_read": ([_vp, _sz, _szp], _i),
    "dt_timeline_mark": ([_vp, _u32], _i),
    "dt_build_flags": ([], _u32),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res


# dt_timeline_record of include/dt.h (48 bytes)
TIMELINE_DTYPE = np.dtype([("grid", np.uint64), ("kind", np.uint32), ("block", np.uint32),
                           ("sm", np.uint32), ("pad", np.uint32), ("t_start", np.uint64),
                           ("t_waited", np.uint64), ("t_end", np.uint64)])
TIMELINE_KINDS = {1: "reduce", 2: "reduce_shift", 3: "copy_bulk", 4: "copy_vec", 5: "copy_shift",
                  6: "copy_2d", 7: "bucket", 8: "bucket_barrier", 9: "barrier", 10: "mark"}


class DtError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {dt_status_string(status)} (status {status})")


def header_symbols() -> list:
    """Names of the functions include/dt.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(dt_\w+)\s*\(", text, re.M)))


def library() -> ctypes.CDLL:
    return _lib


# ------------------------------------------------------------ marshalling
def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return x.data_ptr()


_VP_ARRAY_TYPES: dict = {}


def _ptr_array(xs: Sequence) -> ctypes.Array:
    n = len(xs) or 1
    t = _VP_ARRAY_TYPES.get(n)
    if t is None:                        # building an array type costs more than filling it
        t = _VP_ARRAY_TYPES[n] = ctypes.c_void_p * n
    return t(*[_ptr(x) for x in xs])


def pointer_table(rows: Sequence[Sequence]) -> np.ndarray:
    """rows[t][p] (tensors or device pointers) as a C-contiguous uint64 array
    of shape [T, P]: the layout of the bucket calls' pointer argument.

    Marshalling a nested list costs about 0.3 us per pointer on every call
    (200 gradients of 8 ranks: ~0.5 ms, more than the collective itself).
    Gradient buffers normally stay allocated for the whole run, so build the
    table once and pass it instead of the list; the table holds addresses, not
    references, so the caller keeps the tensors alive."""
    T = len(rows)
    P = len(rows[0]) if T else 0
    if any(len(r) != P for r in rows):
        raise ValueError("pointer_table: every row needs the same number of ranks")
    return np.array([_ptr(x) for r in rows for x in r], dtype=np.uint64).reshape(T, P)


def _table_arg(rows):
    """(keep-alive array, pointer) for a [T][P] pointer argument."""
    if isinstance(rows, np.ndarray):
        a = np.ascontiguousarray(rows, dtype=np.uint64)
    else:
        a = np.array([_ptr(x) for r in rows for x in r], dtype=np.uint64)
    if a.size == 0:
        return a, None
    return a, a.ctypes.data_as(_vpp)


def _sizes_arg(counts):
    a = np.ascontiguousarray(counts, dtype=np.uint64)
    if a.size == 0:
        return a, None
    return a, a.ctypes.data_as(_szp)


def _code(table: dict, v) -> int:
    if isinstance(v, str):
        return table[v]
    try:
        import torch
        if isinstance(v, torch.dtype):
            return {torch.float32: DT_F32, torch.bfloat16: DT_BF16, torch.int32: DT_I32}[v]
    except ImportError:
        pass
    return int(v)


def _stream(stream, device: int | None = None) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, what: str) -> None:
    if st != DT_OK:
        raise DtError(st, what)


# ------------------------------------------------------------- functions
def dt_status_string(status: int) -> str:
    return _lib.dt_status_string(status).decode()


def dt_launch_count() -> int:
    return int(_lib.dt_launch_count())


def dt_build_flags() -> int:
    """DT_BUILD_* bits of the loaded library's flavour (0: the default build)."""
    return int(_lib.dt_build_flags())


def dt_timeline_start(max_records: int) -> None:
    """Start recording the kernel timeline (a DT_TIMELINE=1 build; raises
    DtError DT_ERR_UNSUPPORTED otherwise)."""
    _check(_lib.dt_timeline_start(max_records), "dt_timeline_start")


def dt_timeline_mark(stream=None, tag: int = 0) -> None:
    """A mark on the timeline at this point of the stream (DT_TIMELINE=1 builds)."""
    _check(_lib.dt_timeline_mark(_stream(stream), tag), "dt_timeline_mark")


def dt_timeline_read(max_records: int):
    """(records as a numpy array of TIMELINE_DTYPE, number recorded)."""
    out = np.zeros(max_records, dtype=TIMELINE_DTYPE)
    n = ctypes.c_size_t()
    _check(_lib.dt_timeline_read(out.ctypes.data, max_records, ctypes.byref(n)), "dt_timeline_read")
    return out[:min(n.value, max_records)], n.value


def dt_group_create(world_size: int, cuda_device: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(_lib.dt_group_create(world_size, cuda_device, ctypes.byref(h)), "dt_group_create")
    return h.value


def dt_group_destroy(g: int) -> None:
    _check(_lib.dt_group_destroy(g), "dt_group_destroy")


def dt_group_reset(g: int, stream=None) -> None:
    _check(_lib.dt_group_reset(g, _stream(stream)), "dt_group_reset")


def dt_group_check(g: int) -> int:
    """Returns the status code (does not raise)."""
    return _lib.dt_group_check(g)


def dt_group_error_detail(g: int):
    r, p, gen = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    code = _lib.dt_group_error_detail(g, ctypes.byref(r), ctypes.byref(p), ctypes.byref(gen))
    return code, r.value, p.value, gen.value


def dt_group_size(g: int) -> int:
    return _lib.dt_group_size(g)


def dt_group_generation(g: int) -> int:
    return int(_lib.dt_group_generation(g))


def dt_group_set_timeout_ms(g: int, ms: int) -> None:
    _check(_lib.dt_group_set_timeout_ms(g, ms), "dt_group_set_timeout_ms")


# ---------------------------------------------------- collective calls
# Each collective is a marshaller (Python arguments -> the C call's argument
# tuple) plus the call.  ``prepare`` runs the marshaller once and returns a
# callable that repeats the same C call, for loops that issue one call many
# times with the same buffers.

def _m_allreduce(g: int, rank: int, ins: Sequence, outs: Sequence, count: int, dtype, op,
                 flags: int = 0, stream=None) -> tuple:
    return (g, rank, _ptr_array(ins), _ptr_array(outs), count, _code(DTYPES, dtype),
            _code(OPS, op), flags, _stream(stream))


def _m_reduce_scatter(g: int, rank: int, ins: Sequence, outs: Sequence, recv_count: int, dtype,
                      op, stream=None) -> tuple:
    return (g, rank, _ptr_array(ins), _ptr_array(outs), recv_count, _code(DTYPES, dtype),
            _code(OPS, op), _stream(stream))


def _m_all_gather(g: int, rank: int, ins: Sequence, outs: Sequence, rows: Sequence | None,
                  rows_equal: int, row_bytes: int, flags: int = 0, stream=None) -> tuple:
    rows_arr = None if rows is None else (ctypes.c_size_t * max(len(rows), 1))(*rows)
    return (g, rank, _ptr_array(ins), _ptr_array(outs), rows_arr, rows_equal, row_bytes, flags,
            _stream(stream))


def _m_all_to_all(g: int, rank: int, ins: Sequence, outs: Sequence, chunk_bytes: int,
                  stream=None) -> tuple:
    return (g, rank, _ptr_array(ins), _ptr_array(outs), chunk_bytes, _stream(stream))


def _m_replicate_to_shard(g: int, rank: int, ins: Sequence, outs: Sequence, shard_idx, rows: int,
                          row_bytes: int, stream=None) -> tuple:
    sidx = None if shard_idx is None else (ctypes.c_int * max(len(shard_idx), 1))(*shard_idx)
    return (g, rank, _ptr_array(ins), _ptr_array(outs), sidx, rows, row_bytes, _stream(stream))


def _m_all_gather_into_vec(g: int, rank: int, ins: Sequence, outs: Sequence,
                           rows: Sequence | None, rows_equal: int, row_bytes: int,
                           stream=None) -> tuple:
    """outs[q * P + r] receives rank r's shard on rank q (rank-local: P entries)."""
    rows_arr = None if rows is None else (ctypes.c_size_t * max(len(rows), 1))(*rows)
    return (g, rank, _ptr_array(ins), _ptr_array(outs), rows_arr, rows_equal, row_bytes,
            _stream(stream))


def _m_all_to_all_2d(g: int, rank: int, ins: Sequence, outs: Sequence, R: int, C: int,
                     elem_bytes: int, src_dim: int, dest_dim: int, stream=None) -> tuple:
    return (g, rank, _ptr_array(ins), _ptr_array(outs), R, C, elem_bytes, src_dim, dest_dim,
            _stream(stream))


def _m_bucket_allreduce(g: int, grads, counts: Sequence[int], dtype, op,
                        bucket_cap_bytes: int = 0, stream=None) -> tuple:
    """grads[t][p]: rank p's gradient t (tensor or device pointer), or the
    same as a prepared ``pointer_table``."""
    _, tp = _table_arg(grads)          # the pointer keeps its array alive
    cts, cp = _sizes_arg(counts)
    return (g, tp, cp, cts.size, _code(DTYPES, dtype), _code(OPS, op), bucket_cap_bytes,
            _stream(stream))


def _m_bucket_allreduce_static(world_size: int, grads, counts: Sequence[int], dtype, op,
                               bucket_cap_bytes: int = 0, stream=None) -> tuple:
    """Allocation-free bucket all-reduce: no group, tables in the library's
    fixed device array (see include/dt.h).  grads as dt_bucket_allreduce."""
    _, tp = _table_arg(grads)
    cts, cp = _sizes_arg(counts)
    return (world_size, tp, cp, cts.size, _code(DTYPES, dtype), _code(OPS, op),
            bucket_cap_bytes, _stream(stream))


def _m_barrier(g: int, rank: int = DT_ALL_RANKS, stream=None) -> tuple:
    return (g, rank, _stream(stream))


_MARSHAL: dict = {}


def _entry(name: str, marshal):
    cfn = getattr(_lib, name)

    def call(*args, **kwargs) -> None:
        _check(cfn(*marshal(*args, **kwargs)), name)

    call.__name__ = call.__qualname__ = name
    call.__doc__ = marshal.__doc__
    call.__signature__ = inspect.signature(marshal).replace(return_annotation=None)
    _MARSHAL[call] = (name, marshal)
    return call


dt_allreduce = _entry("dt_allreduce", _m_allreduce)
dt_reduce_scatter = _entry("dt_reduce_scatter", _m_reduce_scatter)
dt_all_gather = _entry("dt_all_gather", _m_all_gather)
dt_all_to_all = _entry("dt_all_to_all", _m_all_to_all)
dt_replicate_to_shard = _entry("dt_replicate_to_shard", _m_replicate_to_shard)
dt_all_gather_into_vec = _entry("dt_all_gather_into_vec", _m_all_gather_into_vec)
dt_all_to_all_2d = _entry("dt_all_to_all_2d", _m_all_to_all_2d)
dt_bucket_allreduce = _entry("dt_bucket_allreduce", _m_bucket_allreduce)
dt_bucket_allreduce_static = _entry("dt_bucket_allreduce_static", _m_bucket_allreduce_static)
dt_barrier = _entry("dt_barrier", _m_barrier)


class Prepared:
    """One collective call with its arguments marshalled once.

    ``prepare(dt.dt_reduce_scatter, g, r, [x], [y], m, "bf16", "avg", stream)``
    converts the arguments as the call itself would (tensors to addresses,
    lists to pointer arrays, names to codes, ``stream=None`` to the current
    stream at this moment) and keeps them; calling the object makes the same C
    call again, raising DtError on a status other than DT_OK.  It holds
    addresses, not tensors: the caller keeps the buffers alive and in place.
    Marshalling costs a few microseconds per call; from P Python threads in
    rank-local mode it is paid under the interpreter lock, where it can take
    more time than the collective (the 4-rank RS+AG step: 141 us per step
    through the per-call functions, 112 us through prepared calls, as fast
    as native threads)."""

    __slots__ = ("name", "_fn", "_args")

    def __init__(self, fn, *args, **kwargs):
        try:
            self.name, marshal = _MARSHAL[fn]
        except (KeyError, TypeError):
            raise ValueError(f"prepare: {fn!r} is not a collective of this module") from None
        cfn = getattr(_lib, self.name)
        types = cfn.argtypes
        vals = marshal(*args, **kwargs)
        # convert plain integers once, so a call passes ready ctypes values
        self._args = tuple(t(v) if isinstance(v, int) and t in (_vp, _i, _u, _sz, _u32) else v
                           for t, v in zip(types, vals))
        self._fn = cfn

    def __call__(self) -> None:
        st = self._fn(*self._args)
        if st != DT_OK:
            raise DtError(st, self.name)


def prepare(fn, *args, **kwargs) -> Prepared:
    return Prepared(fn, *args, **kwargs)


def dt_bucket_plan(counts: Sequence[int], elem_bytes: int, cap_bytes: int):
    T = len(counts)
    cts = (ctypes.c_size_t * max(T, 1))(*counts)
    out = (ctypes.c_size_t * max(T, 1))()
    nb = ctypes.c_size_t()
    _check(_lib.dt_bucket_plan(cts, T, elem_bytes, cap_bytes, out, ctypes.byref(nb)),
           "dt_bucket_plan")
    return [int(out[t]) for t in range(T)], int(nb.value)


def dt_async_begin(g: int, stream=None) -> int:
    """Open an async scope; returns the communication stream handle (int)."""
    cs = ctypes.c_void_p()
    _check(_lib.dt_async_begin(g, _stream(stream), ctypes.byref(cs)), "dt_async_begin")
    return cs.value or 0


def dt_async_end(g: int) -> int:
    w = ctypes.c_void_p()
    _check(_lib.dt_async_end(g, ctypes.byref(w)), "dt_async_end")
    return w.value


def dt_work_wait(work: int, stream=None) -> None:
    _check(_lib.dt_work_wait(work, _stream(stream)), "dt_work_wait")


def dt_work_query(work: int) -> int:
    """DT_OK when finished, DT_NOT_READY otherwise (does not raise for those)."""
    st = _lib.dt_work_query(work)
    if st not in (DT_OK, DT_NOT_READY):
        raise DtError(st, "dt_work_query")
    return st


def dt_work_free(work: int) -> None:
    _check(_lib.dt_work_free(work), "dt_work_free")


def dt_debug_read_window(g: int, stream=None):
    import numpy as np
    P = dt_group_size(g)
    win = np.zeros((P, P), dtype=np.int32)
    _check(_lib.dt_debug_read_window(g, win.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                     _stream(stream)), "dt_debug_read_window")
    return win


def dt_debug_ring_after_barrier(g: int, ins: Sequence, stage: Sequence, outs: Sequence,
                                nbytes: int, stream=None) -> None:
    _check(_lib.dt_debug_ring_after_barrier(g, _ptr_array(ins), _ptr_array(stage),
                                            _ptr_array(outs), nbytes, _stream(stream)),
           "dt_debug_ring_after_barrier")


def dt_debug_barrier_expect(g: int, extra: int, timeout_ms: int, stream=None) -> None:
    _check(_lib.dt_debug_barrier_expect(g, extra, timeout_ms, _stream(stream)),
           "dt_debug_barrier_expect")
