"""DT_LOG=1 makes the library print every launch (kernel, grid, block, shared
memory, stream, attributes) and every bucket plan it builds or reuses to
stderr.  Checked in a child process, since the switch is read once."""
from __future__ import annotations

import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import torch
    from same_device_collective_gb300 import dt
    g = dt.dt_group_create(3, 0)
    xs = [torch.ones(4099, device="cuda") for _ in range(3)]
    outs = [torch.empty_like(x) for x in xs]
    dt.dt_barrier(g)
    dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, outs, 4099, "f32", "sum")
    grads = [[torch.ones(c, device="cuda") for _ in range(3)] for c in (70000, 100, 5)]
    for _ in range(2):
        dt.dt_bucket_allreduce(g, grads, [70000, 100, 5], "f32", "avg", bucket_cap_bytes=1 << 18)
    torch.cuda.synchronize()
    assert dt.dt_group_check(g) == dt.DT_OK
    assert float(outs[2][4098]) == 3.0
    dt.dt_group_destroy(g)
""")


def run(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=300)


def test_dt_log_prints_launches_and_bucket_plans():
    res = run({"DT_LOG": "1"})
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stderr.splitlines() if l.startswith("dt: ")]
    launches = [l for l in lines if l.startswith("dt: launch ")]
    assert any("barrier_kernel" in l and "grid=(1,1,1) block=(96,1,1)" in l for l in launches)
    assert any("reduce_vec_kernel" in l for l in launches)
    assert sum("bucket_kernel" in l for l in launches) == 4      # 2 buckets x 2 calls
    assert all(l.endswith("-> cudaSuccess") for l in launches)
    assert any("bucket plan in slot" in l and "3 tensors x 3 ranks, 2 buckets" in l for l in lines)
    assert any(l.endswith("reused") for l in lines)


def test_no_output_without_dt_log():
    res = run({"DT_LOG": "0"})
    assert res.returncode == 0, res.stderr[-2000:]
    assert not [l for l in res.stderr.splitlines() if l.startswith("dt: ")]


def test_dt_debug_synchronises_every_launch_and_results_hold():
    # DT_DEBUG=1: each launch is followed by a synchronisation of its stream;
    # the same script (barrier, AllReduce, two bucket calls) still succeeds.
    res = run({"DT_DEBUG": "1", "DT_LOG": "0"})
    assert res.returncode == 0, res.stderr[-2000:]


def test_launches_without_programmatic_dependent_launch():
    # DT_PDL=0: every kernel is launched with plain stream ordering; the same
    # script still succeeds.
    res = run({"DT_PDL": "0", "DT_LOG": "1"})
    assert res.returncode == 0, res.stderr[-2000:]
    launches = [l for l in res.stderr.splitlines() if l.startswith("dt: launch ")]
    assert launches and all(l.endswith("-> cudaSuccess") for l in launches)
