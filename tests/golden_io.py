"""Reader for the hand-derived fixtures under tests/golden/ (no oracle code)."""
from __future__ import annotations

from pathlib import Path

import numpy as np

GOLDEN = Path(__file__).resolve().parent / "golden"


def load(path: Path) -> dict:
    rows, idx, val, count, mask = [], [], [], [], []
    meta = {}
    for line in path.read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *rest = line.split()
        if key in ("cols", "stride", "k"):
            meta[key] = int(rest[0])
        elif key == "dtype":
            meta[key] = rest[0]
        elif key == "row":
            rows.append([int(t, 16) for t in rest])
        elif key == "idx":
            idx.append([int(t) for t in rest])
        elif key == "val":
            val.append([int(t, 16) for t in rest])
        elif key == "count":
            count.append(int(rest[0]))
        elif key == "mask":
            mask.append(int(rest[0]))
        else:
            raise ValueError(f"{path.name}: unknown key {key}")
    dtype = meta.get("dtype", "bf16")
    bits = np.uint32 if dtype == "f32" else np.uint16
    return {
        "name": path.stem,
        "dtype": dtype,
        "cols": meta["cols"],
        "stride": meta["stride"],
        "k": meta["k"],
        "logits": np.array(rows, bits),
        "idx": np.array(idx, np.int32),
        "val": np.array(val, bits),
        "count": np.array(count, np.int32),
        "mask": np.array(mask, np.uint32),
    }


def all_fixtures() -> list[dict]:
    return [load(p) for p in sorted(GOLDEN.glob("*.txt"))]
