"""The Python example in README.md runs as written."""
from __future__ import annotations

import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example_runs():
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert blocks, "no python example"
    scope: dict = {}
    exec(compile(blocks[0], "README.md", "exec"), scope)
    torch.cuda.synchronize()
    full, xs = scope["full"], scope["xs"]
    # every rank holds the same gathered tensor; its first shard is the mean of the
    # ranks' first 2048 rows (checked loosely here; the parity tests are exact)
    for q in range(1, len(full)):
        assert torch.equal(full[q], full[0])
    mean = torch.stack([x[:2048].float() for x in xs]).mean(0)
    assert torch.allclose(full[0][:2048].float(), mean, atol=1e-2)
