"""Host logic of bench.py on CPU: multi-rank aggregation over gloo (world
size 2), byte accounting, and the reference arm's JSON line."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 if rank == 0 else 25.0           # rank 1 is the slow one
        ms, gbs = bench.aggregate(local_ms, 1e9, world)
        q.put((rank, ms, gbs))
    finally:
        dist.destroy_process_group()


def test_aggregate_takes_max_time_and_sums_bytes_over_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, gbs in res:
        assert ms == 25.0                                  # slowest rank's time
        assert gbs == pytest.approx(2 * 1e9 / 25e-3 / 1e9)  # both ranks' bytes


def test_step_bytes_is_the_algorithmic_traffic():
    sys.path.insert(0, ROOT)
    import bench
    rs, ag = bench.step_bytes(P=4, rows=8192, cols=4096, es=2)
    n = 8192 * 4096 * 2
    assert rs == 4 * n + n          # read four inputs, write four quarter-size shards
    assert ag == n + 4 * n          # read four shards, write four full outputs


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "5", "--warmup", "3"], capture_output=True, text=True,
                         cwd=ROOT, timeout=300)
    assert out.returncode == 0, out.stderr
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "5", "--warmup", "3"], capture_output=True, text=True,
                         cwd=ROOT, timeout=300, env=env)
    assert out.returncode == 0 and out.stdout.strip() == ""
