"""Seeded random parity: shapes, strides, row offsets, k, plans, formats and
value mixes drawn at random, every result byte-equal to the CPU oracle.

Complements the hand-picked cases: each draw picks rows (1..48), columns
(1..90000, with a bias to the kernels' edges: chunk and span boundaries),
padding, a row base off the 16-byte grid, k, a plan (every bf16 plan, the
fp16 cluster plans, the wide kernel) and a value mix (plain, sprinkled
specials, heavy ties, all-equal rows).  FUZZ_SEED in the environment picks
another sequence; the committed default is fixed."""
from __future__ import annotations

import os

import numpy as np
import pytest

import oracle
from tests.test_gpu_wide import assert_same, gen, gpu_select

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from wide_bf16_row_gb300 import build
    build.build()


SEED = int(os.environ.get("FUZZ_SEED", "20261203"))
CASES = int(os.environ.get("FUZZ_CASES", "60"))
EDGES = (8192, 16384, 16384 * 2, 31040, 49152, 65536)


def _cols(rng) -> int:
    r = rng.random()
    if r < 0.35:
        return int(rng.integers(1, 4097))
    if r < 0.7:
        return int(rng.integers(4097, 90001))
    e = int(rng.choice(EDGES))
    return max(1, e + int(rng.integers(-9, 10)))


def _values(rng, fmt: str, rows: int, cols: int, stride: int, seed: int) -> np.ndarray:
    kind = rng.random()
    if kind < 0.6:
        return gen(fmt, rows, cols, seed, stride, special_frac=float(rng.choice([0.0, 0.001, 0.02])),
                   dup_frac=float(rng.choice([0.0, 0.01, 0.2])))
    bits = np.uint32 if fmt == "f32" else np.uint16
    x = gen(fmt, rows, cols, seed, stride, special_frac=0.0, dup_frac=0.0)
    if kind < 0.8:
        # heavy ties: a handful of values (±0 among them)
        pool = {"bf16": [0x0000, 0x8000, 0x3F80, 0x4000, 0xBF80, 0x7F80],
                "f16": [0x0000, 0x8000, 0x3C00, 0x4000, 0xBC00, 0x7C00],
                "f32": [0x00000000, 0x80000000, 0x3F800000, 0x40000000, 0xBF800000, 0x7F800000]}[fmt]
        x[:, :cols] = rng.choice(np.array(pool, bits), size=(rows, cols))
    else:
        # one value per row (a row of NaN now and then)
        nan = {"bf16": 0x7FC0, "f16": 0x7E00, "f32": 0x7FC00000}[fmt]
        for r in range(rows):
            x[r, :cols] = bits(nan) if rng.random() < 0.2 else x[r, int(rng.integers(0, cols))]
    return x


@pytest.mark.parametrize("case", range(CASES))
def test_random_case(case):
    rng = np.random.default_rng([SEED, case])
    fmt = str(rng.choice(["bf16", "bf16", "bf16", "f16", "f32"]))
    rows = int(rng.integers(1, 49))
    cols = _cols(rng)
    stride = cols + int(rng.choice([0, 0, 1, 3, 8, 17]))
    offset = int(rng.integers(0, 8))
    wide = rng.random() < 0.25
    k = int(rng.integers(65, 1025)) if wide else int(rng.integers(1, 65))
    if fmt == "bf16" and not wide:
        plan = int(rng.choice([0, 1, 2, 4, 8, 16, 32]))
    elif fmt == "f16" and not wide:
        plan = int(rng.choice([0, 1, 2, 4, 8, 16]))
    else:
        plan = int(rng.choice([0, 64]))
    x = _values(rng, fmt, rows, cols, stride, seed=SEED % 100000 + case)
    exp = oracle.topk(x, cols, k, dtype=fmt)
    got = gpu_select(x, cols, k, fmt, plan=plan, offset=offset)
    assert_same(got, exp, f"fuzz case {case}: {fmt} {rows}x{cols} stride {stride} off {offset} k {k} plan {plan}")


def test_no_fault_after_fuzz():
    from wide_bf16_row_gb300 import topk
    assert topk.device_fault() == 0


HEAD_CASES = int(os.environ.get("FUZZ_HEAD_CASES", "16"))


@pytest.mark.parametrize("case", range(HEAD_CASES))
def test_random_head_case(case):
    """The fused draft head on random shapes: rows 1..16, dims of any multiple
    of 8 up to 640, vocabularies around the tile and grid sizes, k 1..64."""
    import torch

    from oracle import head as head_oracle
    from tests.test_gpu_head import _dev, _np
    from wide_bf16_row_gb300 import synth, topk

    rng = np.random.default_rng([SEED, 1000 + case])
    rows = int(rng.integers(1, 17))
    dim = 8 * int(rng.integers(1, 81))
    vocab = int(rng.choice([int(rng.integers(1, 2000)), int(rng.integers(2000, 40000)),
                            128 * int(rng.integers(140, 170)) + int(rng.integers(-3, 4))]))
    k = int(rng.integers(1, 65))
    h = synth.head_inputs(rows, dim, vocab, k, seed=SEED % 100000 + case)
    got = _np(topk.head_topk_bf16(_dev(h.hidden).view(torch.bfloat16), _dev(h.weight).view(torch.bfloat16), k))
    assert_same(got, head_oracle.topk(h.hidden, h.weight, k), f"head fuzz case {case}: {rows}x{dim}x{vocab} k {k}")
