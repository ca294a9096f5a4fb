"""CPU oracle for the exact per-row bf16 top-k -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference arms may import this package.  The product path
(``wide_bf16_row_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``topk_oracle.c`` (plain C, fp64, a stable merge sort
per row); this module only compiles it with gcc and marshals numpy arrays
through ctypes.  The definition it follows is change 3 and the "Exactness"
table of TensorFold PR #713 ("perf(qwen27): a drafted round overlaps its cache
commit with the next draft, and the drafter's attention and top-k use more of
the GPU"); the conventions the pages leave open are listed in the C file's
header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SOURCE = HERE / "topk_oracle.c"


def library_path(mutant: int = 0) -> Path:
    name = "libtopk_oracle.so" if mutant == 0 else f"libtopk_oracle_mutant{mutant}.so"
    return HERE / name


def build(mutant: int = 0, force: bool = False) -> Path:
    """Compile the oracle (or a numbered deliberately-broken mutant of it)."""
    out = library_path(mutant)
    if out.exists() and not force and out.stat().st_mtime >= SOURCE.stat().st_mtime:
        return out
    tmp = out.with_name(out.name + f".tmp{os.getpid()}")
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-shared", "-fPIC", "-pthread",
           f"-DORACLE_MUTANT={mutant}", str(SOURCE), "-o", str(tmp), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


DTYPES = {"bf16": (0, np.uint16), "f16": (1, np.uint16), "f32": (2, np.uint32)}


class Oracle:
    """ctypes handle on one build of the oracle library."""

    def __init__(self, mutant: int = 0):
        self.mutant = mutant
        self._lib = ctypes.CDLL(str(build(mutant)))
        fn = self._lib.oracle_topk
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                       ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                       ctypes.c_void_p, ctypes.c_int32]
        self._fn = fn

    def topk(self, logits: np.ndarray, cols: int, k: int, nthreads: int | None = None, dtype: str = "bf16"):
        """Top-k of every row of ``logits`` (bit patterns of ``dtype``: uint16 for
        "bf16" and "f16", uint32 for "f32"; shape rows x row_stride).

        Returns ``(idx int32[rows,k], val [rows,k] bits of dtype, count int32[rows],
        mask uint32[rows])``.
        """
        code, bits = DTYPES[dtype]
        x = np.ascontiguousarray(logits, dtype=bits)
        if x.ndim != 2:
            raise ValueError("logits must be 2-D (rows x row_stride)")
        rows, stride = x.shape
        idx = np.empty((rows, k), np.int32)
        val = np.empty((rows, k), bits)
        count = np.empty(rows, np.int32)
        mask = np.empty(rows, np.uint32)
        if nthreads is None:
            nthreads = host_cores()
        rc = self._fn(x.ctypes.data, code, rows, cols, stride, k, idx.ctypes.data, val.ctypes.data,
                      count.ctypes.data, mask.ctypes.data, int(nthreads))
        if rc != 0:
            raise RuntimeError(f"oracle_topk failed with status {rc}")
        return idx, val, count, mask


def host_cores() -> int:
    """Cores this process may run on (its affinity mask)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux
        return os.cpu_count() or 1


_default: Oracle | None = None


def topk(logits: np.ndarray, cols: int, k: int, nthreads: int | None = None, dtype: str = "bf16"):
    """Module-level shortcut on the (unmutated) oracle."""
    global _default
    if _default is None:
        _default = Oracle(0)
    return _default.topk(logits, cols, k, nthreads, dtype)
