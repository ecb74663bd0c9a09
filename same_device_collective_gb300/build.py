"""Build libdt.so (the C-ABI collective library) for sm_103a with nvcc.

Each source compiles to an object in parallel, then nvcc links the shared
library next to this file.  The CUDA runtime is linked statically, so the
library only needs the driver at run time.  The rank_local_step program (the
rank-local call pattern from native threads) is linked against it.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build", "dt")
LIB = os.path.join(PKG, "libdt.so")
# rank-local pattern from native threads, linked against libdt.so
STEP_TOOL = os.path.join(PKG, "rank_local_step")

SOURCES = ["dt_group.cpp", "dt_reduce.cu", "dt_reduce_shift.cu", "dt_copy.cu", "dt_bucket.cu",
           "dt_barrier.cu", "dt_static.cu"]
HEADERS = ["dt_internal.h", "dt_group.h", "dt_math.cuh", "dt_device.cuh", "dt_shift.cuh",
           "dt_reduce_shift.h", "dt_timeline.cuh", "dt_timeline.h", "dt_bounds.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# -fmad=false: no multiply-add contraction anywhere (the reductions use
# explicitly rounded adds, divides and multiplies; this keeps it that way).
NVFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-fmad=false", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-Wall", "-I", INCLUDE, "-I", CSRC]
# DT_NVTX=1: every public entry point opens an NVTX range (profiler timelines);
# its objects live in their own folder so the two flavours never mix.
if os.environ.get("DT_NVTX") == "1":
    NVFLAGS.append("-DDT_NVTX")
    BUILD = BUILD + "_nvtx"
# DT_TIMELINE=1: every kernel block records its start, wait and end times
# (dt_timeline_start / dt_timeline_read); its objects live in their own folder.
if os.environ.get("DT_TIMELINE") == "1":
    NVFLAGS.append("-DDT_TIMELINE")
    BUILD = BUILD + "_timeline"
# DT_BOUNDS=1: every data kernel checks each global load and store against the
# extent of its buffer (from the call's arguments); an access outside records
# DT_ERR_INVALID in the group's error word and is skipped.  Own object folder.
if os.environ.get("DT_BOUNDS") == "1":
    NVFLAGS.append("-DDT_BOUNDS")
    BUILD = BUILD + "_bounds"


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdt.so")
    return path


def _stale(target: str, deps: list) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, verbose_ptxas: bool) -> str:
    obj = os.path.join(BUILD, src + ".o")
    deps = [os.path.join(CSRC, src), os.path.join(INCLUDE, "dt.h")] + \
        [os.path.join(CSRC, h) for h in HEADERS]
    if not _stale(obj, deps):
        return obj
    lang = ["-x", "cu"] if src.endswith(".cu") else []
    cmd = [nvcc(), *ARCH, *NVFLAGS, *lang, "-c", os.path.join(CSRC, src), "-o", obj + ".tmp"]
    if verbose_ptxas and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    if verbose_ptxas:
        print(res.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    if force:
        for f in os.listdir(BUILD):
            os.remove(os.path.join(BUILD, f))
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas), SOURCES))
    stamp = LIB + ".objs"            # the objects the library was last linked from
    linked = open(stamp).read() if os.path.exists(stamp) else ""
    if force or _stale(LIB, objs) or linked != "\n".join(objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs,
               "-lpthread", "-ldl", "-lrt"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, LIB)
        with open(stamp, "w") as f:
            f.write("\n".join(objs))
    tool_src = os.path.join(CSRC, "rank_local_step.cpp")
    if force or _stale(STEP_TOOL, [tool_src, LIB, os.path.join(INCLUDE, "dt.h")]):
        tmp = STEP_TOOL + f".tmp{os.getpid()}"
        cmd = [nvcc(), "-O2", "-std=c++17", "-I", INCLUDE, "-x", "c++", tool_src, "-o", tmp,
               "-L", PKG, "-ldt", "-Xlinker", "-rpath,$ORIGIN", "-lpthread"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"rank_local_step build failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, STEP_TOOL)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
