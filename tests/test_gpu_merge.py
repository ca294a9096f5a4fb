"""GPU parity of tf_topk_merge_bf16, the shard-list merge (the merge stage of
TensorFold PR #713, change 3, exposed on its own).

A row's columns are cut into shards (uneven column blocks); each shard's top
k_in list, with indices local to its block, is what tf_topk_bf16 would write
for that block.  Merging them must give the whole row's top k whenever
k_in >= k.  The shard lists here come from the CPU oracle run on each block
(so the GPU merge alone is under test) and, separately, from the GPU's own
per-block calls; the expected row is the oracle on the whole row, byte for
byte."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_same, to_numpy
from wide_bf16_row_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from wide_bf16_row_gb300 import build
    build.build()


def _cuts(cols: int, shards: int, rng) -> list[int]:
    """Uneven column blocks covering [0, cols): sorted interior cut points."""
    inner = np.sort(rng.choice(np.arange(1, cols), size=shards - 1, replace=False)) if shards > 1 else []
    return [0, *[int(c) for c in inner], cols]


def _shard_lists(x: np.ndarray, cols: int, cuts: list[int], k_in: int, source: str):
    """Per-shard lists as stacked arrays [shards, rows, ...] (oracle or GPU)."""
    import torch

    from tests.gpu_util import device_matrix
    from wide_bf16_row_gb300 import topk

    parts = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        block = np.ascontiguousarray(x[:, a:b])
        if source == "oracle":
            parts.append(oracle.topk(block, b - a, k_in))
        else:
            view, keep = device_matrix(block, b - a)
            parts.append(to_numpy(topk.topk_bf16(view, k_in)))
            del keep
    idx = np.stack([p[0] for p in parts]).astype(np.int32)
    val = np.stack([p[1] for p in parts]).astype(np.uint16)
    cnt = np.stack([p[2] for p in parts]).astype(np.int32)
    msk = np.stack([p[3] for p in parts]).astype(np.uint32)
    dev = torch.device("cuda:0")
    return (torch.from_numpy(idx).to(dev), torch.from_numpy(val.view(np.int16)).to(dev),
            torch.from_numpy(cnt).to(dev), torch.from_numpy(msk.view(np.int32)).to(dev))


def _merge(lists, cuts, k):
    from wide_bf16_row_gb300 import topk
    return to_numpy(topk.merge_bf16(*lists, cuts[:-1], k))


CASES = [
    # rows, cols, shards, k, k_in, generator
    (6, 98592, 8, 16, 16, "mixed"),
    (4, 248320, 16, 64, 64, "mixed"),
    (3, 5000, 3, 20, 24, "mixed"),
    (5, 4096, 1, 8, 8, "mixed"),
    (2, 70000, 64, 20, 20, "mixed"),
    (9, 3000, 5, 64, 64, "ties"),
]


def _rows(rows, cols, kind, seed):
    if kind == "mixed":
        return synth.mixed_rows(rows, cols, seed=seed, special_frac=0.01, dup_frac=0.02)
    rng = np.random.default_rng(seed)
    out = np.empty((rows, cols), np.uint16)
    out[0] = 0x3F80                                              # all equal: lowest indices win
    out[1] = rng.integers(0, 2, size=cols, dtype=np.uint16) << np.uint16(15)  # +-0 only
    out[2] = 0x7FC1                                              # all NaN: count 0
    out[3] = np.where(rng.random(cols) < 0.5, 0x4000, 0x3F80)     # two values
    out[4] = 0xFF80                                              # -inf, then a few finite
    out[4, rng.choice(cols, 7, replace=False)] = 0x3F80
    for r in range(5, rows):
        out[r] = synth.round_to_bf16(rng.standard_normal(cols).astype(np.float32))
    return out


@pytest.mark.parametrize("rows,cols,shards,k,k_in,kind", CASES)
@pytest.mark.parametrize("source", ["oracle", "gpu"])
def test_merge_of_shard_lists_equals_whole_row(rows, cols, shards, k, k_in, kind, source):
    rng = np.random.default_rng(cols + shards)
    x = _rows(rows, cols, kind, seed=int(rng.integers(1 << 30)))
    cuts = _cuts(cols, shards, rng)
    got = _merge(_shard_lists(x, cols, cuts, k_in, source), cuts, k)
    assert_same(got, oracle.topk(x, cols, k), f"{rows}x{cols} shards={shards} k={k} k_in={k_in} {source}")


def test_merge_with_shorter_lists_is_the_top_of_their_union():
    """k_in < k: the result is the best k of the entries given (a plain sort of
    their union by score, then global index)."""
    rng = np.random.default_rng(11)
    x = synth.mixed_rows(4, 20000, seed=5, special_frac=0.01, dup_frac=0.05)
    cuts = _cuts(20000, 6, rng)
    k_in, k = 5, 24
    lists = _shard_lists(x, 20000, cuts, k_in, "oracle")
    got = _merge(lists, cuts, k)
    idx, val, cnt, msk = (t.cpu().numpy() for t in lists)
    val = val.view(np.uint16)
    for r in range(4):
        entries = []
        for s in range(len(cuts) - 1):
            for p in range(cnt[s, r]):
                v = float(synth.bf16_to_float(np.array([val[s, r, p]]))[0])
                entries.append((-v, cuts[s] + int(idx[s, r, p]), int(val[s, r, p])))
        entries.sort()
        n = min(k, len(entries))
        assert got[2][r] == n
        assert list(got[0][r, :n]) == [e[1] for e in entries[:n]]
        assert list(got[1][r, :n]) == [e[2] for e in entries[:n]]
        assert all(got[0][r, n:] == -1)
        assert got[3][r] == np.bitwise_or.reduce(msk.view(np.uint32)[:, r])
