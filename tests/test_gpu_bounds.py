"""The bounds-checked flavour of the library (DT_BOUNDS=1 when building).

In that flavour every global load and store of the data kernels is checked
against its buffer's extent as the call's arguments give it; an access
outside is skipped and DT_ERR_INVALID is recorded in the group's error word.
tests/conftest.py turns every recorded access into a test failure, so
`pytest -m gpu` on that build runs the whole GPU suite under the checks.
Here the checker itself is shown to fire: with DT_BOUNDS_TRIM=16 every
destination is recorded 16 bytes short, so the kernels' last stores (inside
the real buffers) are reported and skipped.  Skipped in the default build.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

TESTS = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(TESTS)

CHILD = r"""
import json, sys
import numpy as np, torch
sys.path[:0] = [ROOT, TESTS]
from same_device_collective_gb300 import dt
import oracle
from gpu_util import host, rand_inputs

res = {}
P, n = 4, 4096
xs = rand_inputs(P, n, "bf16", 11)
outs = [torch.full((n,), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
g = dt.dt_group_create(P, 0)
dt.dt_allreduce(g, dt.DT_ALL_RANKS, xs, outs, n, "bf16", "sum")
torch.cuda.synchronize()
code, kernel, buf, off = dt.dt_group_error_detail(g)
want = oracle.allreduce("bf16", "sum", [host(x) for x in xs])
got = [host(o) for o in outs]
res["allreduce"] = dict(
    code=code, kernel=kernel, buf=buf, off=off,
    body=all(np.array_equal(got[r][:n - 8], want[r][:n - 8]) for r in range(P)),
    tail=all(bool((got[r][n - 8:] == 0x40E0).all()) for r in range(P)))
dt.dt_group_destroy(g)

shard = 8192
ins = [torch.randint(0, 255, (shard,), dtype=torch.uint8, device="cuda") for _ in range(P)]
outs = [torch.full((P * shard,), 0xA5, dtype=torch.uint8, device="cuda") for _ in range(P)]
g = dt.dt_group_create(P, 0)
dt.dt_all_gather(g, dt.DT_ALL_RANKS, ins, outs, None, 1, shard)
torch.cuda.synchronize()
code, kernel, buf, off = dt.dt_group_error_detail(g)
want = np.concatenate([x.cpu().numpy() for x in ins])
got = [o.cpu().numpy() for o in outs]
last = slice((P - 1) * shard, P * shard)
res["all_gather"] = dict(
    code=code, kernel=kernel, buf=buf, off=off,
    body=all(np.array_equal(o[:(P - 1) * shard], want[:(P - 1) * shard]) for o in got),
    last=all(bool(((o[last] == want[last]) | (o[last] == 0xA5)).all()) for o in got),
    tail=all(bool((o[-16:] == 0xA5).all()) for o in got))
dt.dt_group_destroy(g)
print("RESULT " + json.dumps(res))
"""


@pytest.fixture(scope="module")
def dt():
    from same_device_collective_gb300 import dt as mod
    assert torch.cuda.is_available()
    if not mod.dt_build_flags() & mod.DT_BUILD_BOUNDS:
        pytest.skip("needs the bounds-checked build (DT_BOUNDS=1 when building)")
    return mod


def test_checker_reports_and_skips_stores_past_a_trimmed_extent(dt):
    env = dict(os.environ, DT_BOUNDS_TRIM="16")
    code = CHILD.replace("ROOT", repr(ROOT)).replace("TESTS", repr(TESTS))
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr[-3000:]
    line = [ln for ln in out.stdout.splitlines() if ln.startswith("RESULT ")][-1]
    res = json.loads(line[len("RESULT "):])

    ar = res["allreduce"]
    assert ar["code"] == dt.DT_ERR_INVALID
    assert dt.BOUNDS_KERNELS[ar["kernel"]] == "reduce"
    assert 16 <= ar["buf"] < 16 + 4                  # an output buffer
    assert ar["off"] == 4096 * 2 - 16                # its last 16-byte vector
    assert ar["body"] and ar["tail"]                 # the rest stored, the last vector skipped

    ag = res["all_gather"]
    assert ag["code"] == dt.DT_ERR_INVALID
    assert dt.BOUNDS_KERNELS[ag["kernel"]] in ("copy_bulk", "copy_vec")
    assert 256 <= ag["buf"] < 256 + 4                # a destination buffer
    assert ag["body"] and ag["last"] and ag["tail"]
