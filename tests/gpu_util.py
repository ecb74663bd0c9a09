"""Helpers shared by the GPU tests: device/host conversion and group fixtures."""
from __future__ import annotations

import contextlib

import numpy as np
import torch

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "i32": torch.int32}
ELEM = {"f32": 4, "bf16": 2, "i32": 4}


def host(t: torch.Tensor) -> np.ndarray:
    """Device tensor -> numpy (bf16 as raw uint16 bits), flattened."""
    t = t.detach().contiguous().cpu().reshape(-1)
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bytes_of(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a).reshape(-1).view(np.uint8)


def rand_inputs(P: int, n: int, dtype: str, seed: int, device="cuda") -> list:
    g = torch.Generator().manual_seed(seed)
    out = []
    for _ in range(P):
        if dtype == "i32":
            x = torch.randint(-2 ** 20, 2 ** 20 + 1, (n,), generator=g, dtype=torch.int32)
        else:
            x = (torch.rand(n, generator=g) * 2 - 1).to(TORCH_DTYPE[dtype])
        out.append(x.to(device))
    return out


def offset_view(n: int, dtype: str, offset_elems: int, device="cuda", fill=None) -> torch.Tensor:
    """A length-n tensor that starts offset_elems into a larger allocation
    (breaks 16-byte alignment when offset_elems * elem % 16 != 0)."""
    base = torch.empty(n + offset_elems + 16, dtype=TORCH_DTYPE[dtype], device=device)
    if fill is not None:
        base.fill_(fill)
    return base[offset_elems:offset_elems + n]


@contextlib.contextmanager
def group(P: int):
    from same_device_collective_gb300 import dt
    g = dt.dt_group_create(P, 0)
    try:
        yield g
    finally:
        torch.cuda.synchronize()
        dt.dt_group_destroy(g)
