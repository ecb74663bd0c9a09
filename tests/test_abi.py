"""CPU checks of the C ABI: the library loads, exports every function that
include/dt.h declares, and its host-only logic (argument checks that need no
device, the bucket plan, status strings) behaves.  No compute call is made."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def dt():
    import __graft_entry__
    __graft_entry__.build()
    from same_device_collective_gb300 import dt as mod
    return mod


def test_library_exports_every_header_symbol(dt):
    names = dt.header_symbols()
    assert len(names) >= 15
    for name in ["dt_group_create", "dt_allreduce", "dt_reduce_scatter", "dt_all_gather",
                 "dt_all_to_all", "dt_bucket_allreduce", "dt_barrier"]:
        assert name in names
    lib = dt.library()
    missing = [n for n in names if not hasattr(lib, n)]
    assert missing == []


def test_binding_has_the_c_names(dt):
    for name in dt.header_symbols():
        assert callable(getattr(dt, name)), name


def test_status_strings(dt):
    for code in range(9):
        assert dt.dt_status_string(code) != "unknown status"
    assert dt.dt_status_string(99) == "unknown status"


def test_null_group_is_invalid_without_touching_a_device(dt):
    lib = dt.library()
    assert lib.dt_allreduce(None, -1, None, None, 0, 0, 0, 0, None) == dt.DT_ERR_INVALID
    assert lib.dt_reduce_scatter(None, -1, None, None, 0, 0, 0, None) == dt.DT_ERR_INVALID
    assert lib.dt_all_gather(None, -1, None, None, None, 0, 0, 0, None) == dt.DT_ERR_INVALID
    assert lib.dt_all_to_all(None, -1, None, None, 0, None) == dt.DT_ERR_INVALID
    assert lib.dt_bucket_allreduce(None, None, None, 0, 0, 0, 0, None) == dt.DT_ERR_INVALID
    assert lib.dt_barrier(None, -1, None) == dt.DT_ERR_INVALID
    assert lib.dt_group_destroy(None) == dt.DT_ERR_INVALID
    assert lib.dt_group_check(None) == dt.DT_ERR_INVALID
    assert lib.dt_group_size(None) == 0
    assert lib.dt_group_create(0, 0, None) == dt.DT_ERR_INVALID
    h = ctypes.c_void_p()
    assert lib.dt_group_create(17, 0, ctypes.byref(h)) == dt.DT_ERR_INVALID
    assert lib.dt_group_create(0, 0, ctypes.byref(h)) == dt.DT_ERR_INVALID


def test_bucket_plan_host_logic_matches_oracle(dt):
    from same_device_collective_gb300 import workloads
    rng = np.random.default_rng(5)
    cases = [([10, 10, 10], 2, 40), ([30, 5, 30], 2, 40), ([], 2, 40), ([0, 100, 1], 2, 10),
             (workloads.bucket_counts(), 2, workloads.BUCKET_CAP_BYTES),
             ([int(c) for c in rng.integers(0, 5000, 500)], 4, 4096)]
    for counts, es, cap in cases:
        assert dt.dt_bucket_plan(counts, es, cap) == oracle.bucket_plan(counts, es, cap)
    with pytest.raises(dt.DtError):
        dt.dt_bucket_plan([1], 0, 10)
    with pytest.raises(dt.DtError):
        dt.dt_bucket_plan([1], 2, 0)


def test_launch_counter_starts_at_zero_without_work(dt):
    assert dt.dt_launch_count() >= 0


def test_pointer_table_marshals_tensors_and_addresses(dt):
    import torch
    ts = [[torch.empty(4), 1234, torch.empty(2)], [16, torch.empty(1), 0]]
    tab = dt.pointer_table(ts)
    assert tab.dtype == np.uint64 and tab.shape == (2, 3) and tab.flags["C_CONTIGUOUS"]
    assert tab[0, 0] == ts[0][0].data_ptr() and tab[0, 1] == 1234 and tab[1, 2] == 0
    assert tab[1, 1] == ts[1][1].data_ptr()
    assert dt.pointer_table([]).shape == (0, 0)
    with pytest.raises(ValueError):
        dt.pointer_table([[1, 2], [3]])
    # the bucket calls take either form; with no group both fail validation alike
    lib_status = []
    for arg in (ts, tab):
        with pytest.raises(dt.DtError) as e:
            dt.dt_bucket_allreduce(None, arg, [4, 1], "f32", "sum", stream=0)
        lib_status.append(e.value.status)
    assert lib_status == [dt.DT_ERR_INVALID] * 2


def test_nvtx_flavour_compiles(tmp_path):
    # DT_NVTX=1 builds wrap every entry point in an NVTX range; the host
    # translation unit must compile that way too (compiled to a scratch
    # object here, so the in-tree library is left as it is).
    import os
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    from same_device_collective_gb300 import build as b
    cmd = [b.nvcc(), *b.ARCH, "-O1", "-std=c++17", "-Xcompiler", "-fPIC", "-DDT_NVTX",
           "-I", os.path.join(root, "include"), "-I", b.CSRC, "-c",
           os.path.join(b.CSRC, "dt_group.cpp"), "-o", str(tmp_path / "g.o")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr


def test_prepared_calls_make_the_same_call_as_the_functions(dt):
    # With a null group every entry point returns DT_ERR_INVALID before it
    # looks at anything else, so the marshalled arguments can be exercised
    # without a device (explicit stream handles; pointers are never read).
    cases = [(dt.dt_allreduce, (None, -1, [16, 32], [48, 64], 16, "f32", "sum", 0, 7)),
             (dt.dt_reduce_scatter, (None, -1, [16], [32], 4, "bf16", "avg", 7)),
             (dt.dt_all_gather, (None, -1, [16], [32], [3], 0, 16, 0, 7)),
             (dt.dt_all_to_all, (None, -1, [16], [32], 16, 7)),
             (dt.dt_all_to_all_2d, (None, -1, [16], [32], 4, 4, 2, 0, 1, 7)),
             (dt.dt_replicate_to_shard, (None, -1, [16], [32], None, 4, 16, 7)),
             (dt.dt_all_gather_into_vec, (None, -1, [16], [32], None, 1, 16, 7)),
             (dt.dt_barrier, (None, -1, 7)),
             (dt.dt_bucket_allreduce, (None, [[16, 32]], [4], "f32", "avg", 0, 7))]
    for fn, args in cases:
        p = dt.prepare(fn, *args)
        assert p.name == fn.__name__
        for _ in range(2):                                  # reusable
            with pytest.raises(dt.DtError) as e:
                p()
            assert e.value.status == dt.DT_ERR_INVALID, fn.__name__
        with pytest.raises(dt.DtError) as e:
            fn(*args)
        assert e.value.status == dt.DT_ERR_INVALID, fn.__name__
    with pytest.raises(ValueError):
        dt.prepare(dt.dt_status_string, 0)
    with pytest.raises(ValueError):
        dt.prepare(print, 0)


def test_timeline_is_unsupported_in_the_default_build(dt):
    # Only a DT_TIMELINE=1 build records the kernel timeline; the default one
    # answers without touching a device.
    lib = dt.library()
    assert lib.dt_timeline_start(16) == dt.DT_ERR_UNSUPPORTED
    n = ctypes.c_size_t()
    assert lib.dt_timeline_read(None, 0, ctypes.byref(n)) == dt.DT_ERR_UNSUPPORTED
    assert lib.dt_timeline_mark(None, 3) == dt.DT_ERR_UNSUPPORTED
    assert dt.TIMELINE_DTYPE.itemsize == 48


def test_timeline_flavour_compiles(tmp_path):
    # DT_TIMELINE=1 builds instrument the kernels; the host unit and the
    # smallest kernel unit must compile that way (scratch objects only).
    import os
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    from same_device_collective_gb300 import build as b
    for src, lang in (("dt_group.cpp", []), ("dt_barrier.cu", ["-x", "cu"])):
        cmd = [b.nvcc(), *b.ARCH, "-O1", "-std=c++17", "-Xcompiler", "-fPIC", "-DDT_TIMELINE",
               "-I", os.path.join(root, "include"), "-I", b.CSRC, *lang, "-c",
               os.path.join(b.CSRC, src), "-o", str(tmp_path / (src + ".o"))]
        res = subprocess.run(cmd, capture_output=True, text=True)
        assert res.returncode == 0, res.stderr


def test_build_flags_name_the_flavour(dt):
    # dt_build_flags reports the instrumented flavour: the timeline calls
    # answer DT_ERR_UNSUPPORTED exactly when DT_BUILD_TIMELINE is clear.
    lib = dt.library()
    flags = dt.dt_build_flags()
    assert flags & ~(dt.DT_BUILD_NVTX | dt.DT_BUILD_TIMELINE | dt.DT_BUILD_BOUNDS) == 0
    n = ctypes.c_size_t()
    unsupported = lib.dt_timeline_read(None, 0, ctypes.byref(n)) == dt.DT_ERR_UNSUPPORTED
    assert unsupported == (not flags & dt.DT_BUILD_TIMELINE)


def test_bounds_flavour_compiles(tmp_path):
    # DT_BOUNDS=1 builds check every kernel access against its buffer; the
    # host unit (extents from the arguments) and the bucket kernel unit must
    # compile that way (scratch objects only).
    import os
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    from same_device_collective_gb300 import build as b
    for src, lang in (("dt_group.cpp", []), ("dt_bucket.cu", ["-x", "cu"])):
        cmd = [b.nvcc(), *b.ARCH, "-O1", "-std=c++17", "-Xcompiler", "-fPIC", "-DDT_BOUNDS",
               "-I", os.path.join(root, "include"), "-I", b.CSRC, *lang, "-c",
               os.path.join(b.CSRC, src), "-o", str(tmp_path / (src + ".o"))]
        res = subprocess.run(cmd, capture_output=True, text=True)
        assert res.returncode == 0, res.stderr


C_CALLER = r"""
#include <stdio.h>
#include <string.h>
#include "dt.h"

int main(void)
{
    dt_group_t g = 0;
    /* calls that need no device: argument checks, strings, flags */
    if (dt_group_create(0, 0, &g) != DT_ERR_INVALID) return 1;
    if (dt_group_destroy(0) != DT_ERR_INVALID) return 2;
    if (strlen(dt_status_string(DT_OK)) == 0) return 3;
    /* 2-byte elements, 40-byte cap: 20 B | 40 B | 60 B (over the cap, alone) */
    size_t counts[3] = {10, 20, 30}, bucket_of[3] = {9, 9, 9}, n_buckets = 0;
    if (dt_bucket_plan(counts, 3, 2, 40, bucket_of, &n_buckets) != DT_OK) return 4;
    if (n_buckets != 3 || bucket_of[0] != 0 || bucket_of[1] != 1 || bucket_of[2] != 2) return 5;
    printf("%u\n", dt_build_flags());
    return 0;
}
"""


def test_header_is_plain_c_and_links(tmp_path):
    # include/dt.h is a C header: a C11 program that includes it compiles
    # with every warning an error, links against libdt.so and calls the
    # entry points that need no device.
    import os
    import subprocess
    from same_device_collective_gb300 import build as b
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    pkg = os.path.dirname(b.LIB)
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror",
           "-I", os.path.join(root, "include"), str(src), "-o", str(exe),
           "-L", pkg, "-ldt", "-Wl,-rpath," + pkg]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, (run.returncode, run.stderr)
    assert run.stdout.strip().isdigit()
