import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs on a GB300)")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.lib()
    return oracle


# ---- bounds-checked library builds (DT_BOUNDS=1) --------------------------
# In that flavour every kernel access outside its buffer is skipped and
# recorded as DT_ERR_INVALID in the group's error word.  Every group the GPU
# tests create is looked at when it is destroyed and after each test, so a
# whole `pytest -m gpu` run on that build fails on any out-of-bounds access.
_BOUNDS_HITS: list = []
_LIVE_GROUPS: set = set()


def _bounds_build() -> bool:
    try:
        from same_device_collective_gb300 import dt
    except ImportError:
        return False
    return bool(dt.dt_build_flags() & dt.DT_BUILD_BOUNDS)


def _bounds_hit(dt, g):
    code, rank, peer, gen = dt.dt_group_error_detail(g)
    if code == dt.DT_ERR_INVALID:
        return (dt.BOUNDS_KERNELS.get(rank, rank), peer, gen)
    return None


@pytest.fixture(scope="session", autouse=True)
def _watch_bounds():
    if os.environ.get("DT_BOUNDS_TRIM") or not _bounds_build():
        yield
        return
    from same_device_collective_gb300 import dt
    create, destroy = dt.dt_group_create, dt.dt_group_destroy

    def checked_create(*a, **k):
        g = create(*a, **k)
        _LIVE_GROUPS.add(g)
        return g

    def checked_destroy(g):
        if g in _LIVE_GROUPS:
            _LIVE_GROUPS.discard(g)
            hit = _bounds_hit(dt, g)
            if hit:
                _BOUNDS_HITS.append(hit)
        destroy(g)

    dt.dt_group_create, dt.dt_group_destroy = checked_create, checked_destroy
    yield
    dt.dt_group_create, dt.dt_group_destroy = create, destroy


@pytest.fixture(autouse=True)
def _no_bounds_hits(_watch_bounds):
    yield
    if not _LIVE_GROUPS and not _BOUNDS_HITS:
        return
    from same_device_collective_gb300 import dt
    hits = list(_BOUNDS_HITS)
    _BOUNDS_HITS.clear()
    hits += [h for h in (_bounds_hit(dt, g) for g in list(_LIVE_GROUPS)) if h]
    assert not hits, f"out-of-bounds accesses (kernel, buffer, byte offset): {hits}"
