"""Build the CUDA library ``libtf_topk.so`` in-tree for sm_103a.

``python -m wide_bf16_row_gb300.build`` (or ``__graft_entry__.build()``) runs
nvcc once; the result sits next to this file, where the binding loads it.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
SOURCES = [PKG / "csrc" / "tf_topk.cu", PKG / "csrc" / "tf_topk_head.cu", PKG / "csrc" / "tf_topk_f32.cu"]
HEADERS = [ROOT / "include" / "tf_topk.h"]
LIBRARY = PKG / "libtf_topk.so"
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def compile_command(src: Path, obj: Path, defines: tuple[str, ...] = ()) -> list[str]:
    return [nvcc(), "-O3", "-std=c++17", ARCH, "-lineinfo", "-Xcompiler", "-fPIC", "-c",
            *[f"-D{d}" for d in defines], "-I", str(ROOT / "include"), "-o", str(obj), str(src)]


def link_command(objs: list[Path], out: Path) -> list[str]:
    return [nvcc(), ARCH, "-shared", "-o", str(out), *map(str, objs)]


def up_to_date() -> bool:
    if not LIBRARY.exists():
        return False
    t = LIBRARY.stat().st_mtime
    return all(p.stat().st_mtime <= t for p in SOURCES + HEADERS)


def build(force: bool = False, verbose: bool = False) -> Path:
    if up_to_date() and not force:
        return LIBRARY
    return _build_library(LIBRARY, (), verbose)


def build_variant(name: str, defines: tuple[str, ...]) -> Path:
    """A separate library ``libtf_topk_<name>.so`` compiled with extra macros
    (test builds, e.g. a forced wait timeout); the product library is untouched."""
    out = PKG / f"libtf_topk_{name}.so"
    if out.exists() and all(p.stat().st_mtime <= out.stat().st_mtime for p in SOURCES + HEADERS):
        return out
    return _build_library(out, defines, False)


def _build_library(library: Path, defines: tuple[str, ...], verbose: bool) -> Path:
    tmp = library.with_name(f"{library.name}.tmp{os.getpid()}")
    objs = [library.with_name(f"{library.stem}_{src.stem}.tmp{os.getpid()}.o") for src in SOURCES]
    cmds = [compile_command(src, obj, defines) for src, obj in zip(SOURCES, objs)]
    if verbose:
        for cmd in cmds:
            print(" ".join(cmd), file=sys.stderr)
    try:
        # the translation units compile side by side, then one link
        with ThreadPoolExecutor(max_workers=len(cmds)) as pool:
            for result in pool.map(lambda c: subprocess.run(c, check=True), cmds):
                pass
        subprocess.run(link_command(objs, tmp), check=True)
        os.replace(tmp, library)
    finally:
        for obj in objs:
            if obj.exists():
                obj.unlink()
    return library


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(LIBRARY)
