"""Helpers for the GPU parity tests: place a uint16 matrix on the device (with a
chosen element offset, so the row base can be misaligned), call the CUDA path
through the C ABI, bring the four outputs back as numpy arrays."""
from __future__ import annotations

import numpy as np


def device_matrix(x: np.ndarray, cols: int, offset: int = 0, device: str = "cuda:0"):
    """A (rows, cols) int16 CUDA view of ``x`` (rows x row_stride) starting ``offset``
    elements into a fresh buffer."""
    import torch

    rows, stride = x.shape
    flat = torch.empty(offset + rows * stride + 8, dtype=torch.int16, device=device)
    flat.fill_(0x7FC0)  # NaN pattern around the matrix: never read
    flat[offset: offset + rows * stride] = torch.from_numpy(np.ascontiguousarray(x).view(np.int16).ravel()).to(device)
    return flat.as_strided((rows, cols), (stride, 1), offset), flat


def to_numpy(res):
    import torch

    idx, val, count, mask = res
    torch.cuda.synchronize()
    return (idx.cpu().numpy(), val.view(torch.int16).cpu().numpy().view(np.uint16),
            count.cpu().numpy(), mask.cpu().numpy().view(np.uint32))


def gpu_topk(x: np.ndarray, cols: int, k: int, plan: int = 0, offset: int = 0):
    from wide_bf16_row_gb300 import topk

    view, _keep = device_matrix(x, cols, offset)
    res = topk.topk_bf16(view, k, plan=plan)
    out = to_numpy(res)
    del _keep
    return out


def assert_same(got, exp, what: str = ""):
    names = ("idx", "val", "count", "mask")
    for g, e, n in zip(got, exp, names):
        if not np.array_equal(g, e):
            bad = np.argwhere(g != e)
            first = tuple(bad[0]) if len(bad) else None
            raise AssertionError(f"{what}: {n} differs at {len(bad)} places, first {first}: "
                                 f"got {g[first] if first is not None else None} "
                                 f"expected {e[first] if first is not None else None}")
