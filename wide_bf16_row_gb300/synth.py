"""Seeded synthetic bf16 logit matrices for the tests and the benchmark.

This module holds input generation only -- no part of the top-k method.  Both
the CUDA path's tests and the CPU oracle's tests draw their inputs from here.

Every workload is a ``Workload``: a ``rows x row_stride`` uint16 array of bf16
bit patterns (columns ``[cols, row_stride)`` are padding), plus ``cols`` and
``k``.  Values are drawn in float32 from numpy's PCG64 generator and rounded to
bf16 with round-to-nearest-even.  The shapes and value mixes follow the draft
head of TensorFold PR #713 ("perf(qwen27): ... top-k use more of the GPU",
change 3: 15 rows x 98592 columns; the "Exactness" table: widths 4096 to
248320 with ties, both zeros, NaN, infinities and padded strides).  Real
draft-head logits need model weights, so these seeded rows stand in for them.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass

import numpy as np

BF16_POS_INF = 0x7F80
BF16_NEG_INF = 0xFF80
BF16_NEG_ZERO = 0x8000


@dataclass
class Workload:
    name: str
    logits: np.ndarray  # uint16 [rows, row_stride]
    cols: int
    k: int

    @property
    def rows(self) -> int:
        return self.logits.shape[0]

    @property
    def row_stride(self) -> int:
        return self.logits.shape[1]

    def algorithmic_bytes(self) -> int:
        """Bytes one call must move: the valid columns read, the outputs written."""
        return self.rows * self.cols * 2 + self.rows * self.k * 6 + self.rows * 8


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest, ties to even (finite input)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_to_float(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_rows(rng: np.random.Generator, rows: int, cols: int, sigma: float) -> np.ndarray:
    out = np.empty((rows, cols), np.uint16)
    block = max(1, (1 << 24) // max(cols, 1))
    for r0 in range(0, rows, block):
        r1 = min(rows, r0 + block)
        z = rng.standard_normal((r1 - r0, cols), dtype=np.float32)
        z *= np.float32(sigma)
        out[r0:r1] = round_to_bf16(z)
    return out


def _duplicate(rng: np.random.Generator, vals: np.ndarray, frac: float) -> None:
    """Set ``frac`` of each row's entries to the value of another random column."""
    rows, cols = vals.shape
    n = int(round(cols * frac))
    if n == 0 or cols < 2:
        return
    for r in range(rows):
        dst = rng.choice(cols, size=n, replace=False)
        src = rng.integers(0, cols, size=n)
        vals[r, dst] = vals[r, src]


def _pad(rng: np.random.Generator, vals: np.ndarray, row_stride: int) -> np.ndarray:
    rows, cols = vals.shape
    if row_stride == cols:
        return np.ascontiguousarray(vals)
    out = rng.integers(0, 1 << 16, size=(rows, row_stride), dtype=np.uint16)  # garbage pad
    out[:, :cols] = vals
    return out


def _nan_bits(rng: np.random.Generator, n: int) -> np.ndarray:
    sign = rng.integers(0, 2, size=n, dtype=np.uint16) << np.uint16(15)
    payload = rng.integers(1, 0x80, size=n, dtype=np.uint16)
    return (sign | np.uint16(0x7F80) | payload).astype(np.uint16)


def normal(rows: int, cols: int, k: int, sigma: float = 1.0, seed: int = 0,
           row_stride: int | None = None, dup_frac: float = 0.0, name: str | None = None) -> Workload:
    rng = np.random.default_rng(seed)
    vals = _normal_rows(rng, rows, cols, sigma)
    _duplicate(rng, vals, dup_frac)
    stride = cols if row_stride is None else row_stride
    return Workload(name or f"{rows}x{cols}_k{k}", _pad(rng, vals, stride), cols, k)


def config_draft_single(seed: int = 0) -> Workload:
    """1 row x 4096 columns, k = 8, N(0, 1), packed."""
    return normal(1, 4096, 8, sigma=1.0, seed=seed, name="1x4096_k8")


def config_draft_head(seed: int = 1) -> Workload:
    """15 rows x 98592 columns, k = 16, N(0, 3), 1% of entries copied from another column."""
    return normal(15, 98592, 16, sigma=3.0, seed=seed, dup_frac=0.01, name="15x98592_k16")


def config_specials(seed: int = 2, rows: int = 16, cols: int = 248320, row_stride: int = 248384,
                    k: int = 64, nan_row: int = 3, zero_row: int = 7) -> Workload:
    """Padded rows with NaN, +-inf and +-0 mixed in; one all-NaN row, one all-zero row.

    Per row: 0.1% NaN (random payload, either sign), 0.1% +inf, 0.1% -inf,
    1% exact zeros (half +0, half -0), the rest N(0, 2).  The padding columns
    hold random bits, NaN and inf patterns included.
    """
    rng = np.random.default_rng(seed)
    vals = _normal_rows(rng, rows, cols, 2.0)
    n_nan = max(1, cols // 1000)
    n_inf = max(1, cols // 1000)
    n_zero = max(2, cols // 100)
    for r in range(rows):
        pos = rng.permutation(cols)[: n_nan + 2 * n_inf + n_zero]
        a, b, c = n_nan, n_nan + n_inf, n_nan + 2 * n_inf
        vals[r, pos[:a]] = _nan_bits(rng, a)
        vals[r, pos[a:b]] = BF16_POS_INF
        vals[r, pos[b:c]] = BF16_NEG_INF
        zs = pos[c:]
        vals[r, zs[: len(zs) // 2]] = 0
        vals[r, zs[len(zs) // 2:]] = BF16_NEG_ZERO
    if 0 <= nan_row < rows:
        vals[nan_row] = _nan_bits(rng, cols)
    if 0 <= zero_row < rows:
        vals[zero_row] = rng.integers(0, 2, size=cols, dtype=np.uint16) << np.uint16(15)
    return Workload(f"{rows}x{cols}_k{k}_stride{row_stride}_specials", _pad(rng, vals, row_stride),
                    cols, k)


def config_draft_window(seed: int = 3, rows: int = 256, cols: int = 248320, k: int = 20,
                        spikes: int = 5) -> Workload:
    """Rows of N(0, 4) with a Gumbel spike (20 + 4 G) on ``spikes`` random columns per row."""
    rng = np.random.default_rng(seed)
    vals = _normal_rows(rng, rows, cols, 4.0)
    for r in range(rows):
        pos = rng.choice(cols, size=spikes, replace=False)
        u = rng.random(spikes)
        u = np.clip(u, 1e-12, 1 - 1e-12)
        g = -np.log(-np.log(u))
        vals[r, pos] = round_to_bf16((20.0 + 4.0 * g).astype(np.float32))
    return Workload(f"{rows}x{cols}_k{k}", vals, cols, k)


def config_masked_window(seed: int = 4, rows: int = 256, cols: int = 248320, k: int = 20) -> Workload:
    """The 256 x 248320 rows with a tenth of each row's columns masked to -inf
    (a sampling mask over the vocabulary)."""
    return Workload(f"{rows}x{cols}_k{k}_masked", masked_rows(rows, cols, seed, mask_frac=0.1), cols, k)


SWEEP_WIDTHS = (4096, 32768, 98592, 151936, 248320)
SWEEP_ROWS = (1, 4, 15, 64, 1024)
SWEEP_KS = (1, 8, 20, 64)


def sweep_seed(width: int, rows: int, k: int) -> int:
    h = hashlib.sha256(f"{width}x{rows}k{k}".encode()).digest()
    return int.from_bytes(h[:4], "little")


def config_sweep(width: int, rows: int, k: int) -> Workload:
    """N(0, 2) with 0.5% copied values; row stride = width rounded up to 64 (garbage pad)."""
    stride = (width + 63) // 64 * 64
    return normal(rows, width, k, sigma=2.0, seed=sweep_seed(width, rows, k), row_stride=stride,
                  dup_frac=0.005, name=f"sweep_{rows}x{width}_k{k}")


NAMED = {
    "1x4096_k8": config_draft_single,
    "15x98592_k16": config_draft_head,
    "16x248320_k64_specials": config_specials,
    "256x248320_k20": config_draft_window,
}


def special_alphabet() -> np.ndarray:
    """bf16 patterns for -inf, -1, -min subnormal, -0, +0, +min subnormal, +1, +inf, NaN."""
    return np.array([0xFF80, 0xBF80, 0x8001, 0x8000, 0x0000, 0x0001, 0x3F80, 0x7F80, 0x7FC0],
                    dtype=np.uint16)


def mixed_rows(rows: int, cols: int, seed: int, row_stride: int | None = None,
               special_frac: float = 0.05, dup_frac: float = 0.02, sigma: float = 2.0) -> np.ndarray:
    """Normal rows sprinkled with every special pattern, copies and subnormals."""
    rng = np.random.default_rng(seed)
    vals = _normal_rows(rng, rows, cols, sigma)
    _duplicate(rng, vals, dup_frac)
    n = int(cols * special_frac)
    if n:
        extra = np.concatenate([special_alphabet(), np.array([0xFFC1, 0x7F81, 0x0080, 0x807F],
                                                              dtype=np.uint16)])
        for r in range(rows):
            pos = rng.choice(cols, size=n, replace=False)
            vals[r, pos] = extra[rng.integers(0, len(extra), size=n)]
    stride = cols if row_stride is None else row_stride
    return _pad(rng, vals, stride)



def masked_rows(rows: int, cols: int, seed: int, mask_frac: float = 0.1, tail: int = 0,
                plus_inf_frac: float = 0.0, row_stride: int | None = None, fmt: str = "bf16") -> np.ndarray:
    """Masked logits: normal rows (sigma 4) with ``mask_frac`` of each row's
    columns set to -inf at random, the last ``tail`` columns -inf (a padded
    vocabulary), and ``plus_inf_frac`` of the columns +inf.  No NaN.  ``fmt``
    "bf16" or "f16" (uint16 bit patterns) or "f32" (uint32); padding is
    random bits."""
    rng = np.random.default_rng(seed)
    if fmt == "bf16":
        vals = _normal_rows(rng, rows, cols, 4.0)
        ninf, pinf = 0xFF80, 0x7F80
    elif fmt == "f16":
        vals = (rng.standard_normal((rows, cols)) * 4.0).astype(np.float16).view(np.uint16)
        ninf, pinf = 0xFC00, 0x7C00
    else:
        vals = (rng.standard_normal((rows, cols)) * 4.0).astype(np.float32).view(np.uint32)
        ninf, pinf = 0xFF800000, 0x7F800000
    vals[rng.random((rows, cols)) < mask_frac] = ninf
    if tail:
        vals[:, max(0, cols - tail):] = ninf
    if plus_inf_frac:
        vals[rng.random((rows, cols)) < plus_inf_frac] = pinf
    stride = cols if row_stride is None else row_stride
    if fmt != "f32":
        return _pad(rng, vals, stride)
    if stride == cols:
        return np.ascontiguousarray(vals)
    out = rng.integers(0, 1 << 32, size=(rows, stride), dtype=np.uint32)
    out[:, :cols] = vals
    return out

# ---------------------------------------------------------------- fp16 and fp32 rows

def special_alphabet_f16() -> np.ndarray:
    """fp16 patterns for -inf, -max, -1, -min subnormal, -0, +0, +min subnormal,
    +1, +max, +inf and two NaNs (quiet positive, signalling-style negative)."""
    return np.array([0xFC00, 0xFBFF, 0xBC00, 0x8001, 0x8000, 0x0000, 0x0001, 0x3C00, 0x7BFF, 0x7C00,
                     0x7E00, 0xFC01], dtype=np.uint16)


def special_alphabet_f32() -> np.ndarray:
    """fp32 patterns for -inf, -max, -1, -min subnormal, -0, +0, +min subnormal,
    1, the next float above 1 (differs only in the low half), +max, +inf and
    two NaNs."""
    return np.array([0xFF800000, 0xFF7FFFFF, 0xBF800000, 0x80000001, 0x80000000, 0x00000000, 0x00000001,
                     0x3F800000, 0x3F800001, 0x7F7FFFFF, 0x7F800000, 0x7FC00000, 0xFF800001],
                    dtype=np.uint32)


def mixed_rows_f16(rows: int, cols: int, seed: int, row_stride: int | None = None,
                   special_frac: float = 0.05, dup_frac: float = 0.02, sigma: float = 2.0) -> np.ndarray:
    """fp16 bit patterns (uint16): normal rows rounded to fp16, sprinkled with
    the fp16 specials, copies and random subnormals; padding is random bits."""
    rng = np.random.default_rng(seed)
    vals = (rng.standard_normal((rows, cols)) * sigma).astype(np.float16).view(np.uint16)
    _duplicate(rng, vals, dup_frac)
    n = int(cols * special_frac)
    if n:
        alpha = special_alphabet_f16()
        for r in range(rows):
            pos = rng.choice(cols, size=n, replace=False)
            pick = alpha[rng.integers(0, len(alpha), size=n)]
            sub = rng.integers(1, 0x400, size=n, dtype=np.uint16) | (rng.integers(0, 2, size=n, dtype=np.uint16) << np.uint16(15))
            vals[r, pos] = np.where(rng.random(n) < 0.3, sub, pick)
    stride = cols if row_stride is None else row_stride
    return _pad(rng, vals, stride)


def mixed_rows_f32(rows: int, cols: int, seed: int, row_stride: int | None = None,
                   special_frac: float = 0.05, dup_frac: float = 0.02, sigma: float = 2.0) -> np.ndarray:
    """fp32 bit patterns (uint32): normal rows, sprinkled with the fp32
    specials, copies, near-ties that differ only in the low 16 bits, and
    subnormals; padding is random bits."""
    rng = np.random.default_rng(seed)
    vals = (rng.standard_normal((rows, cols)) * sigma).astype(np.float32).view(np.uint32)
    _duplicate(rng, vals, dup_frac)
    n = int(cols * special_frac)
    if n:
        alpha = special_alphabet_f32()
        for r in range(rows):
            pos = rng.choice(cols, size=n, replace=False)
            pick = alpha[rng.integers(0, len(alpha), size=n)]
            near = (vals[r, rng.integers(0, cols, size=n)] ^ rng.integers(1, 1 << 16, size=n, dtype=np.uint32))
            vals[r, pos] = np.where(rng.random(n) < 0.4, near, pick)
    stride = cols if row_stride is None else row_stride
    if stride == cols:
        return np.ascontiguousarray(vals)
    out = rng.integers(0, 1 << 32, size=(rows, stride), dtype=np.uint32)
    out[:, :cols] = vals
    return out


def ranked_lists(rows: int, k: int, seed: int) -> tuple[np.ndarray, np.ndarray]:
    """Lists shaped like a top-k's output, for the step that consumes them:
    ``(val uint16 [rows, k], count int32 [rows])``, each row's first ``count``
    entries best first with NaN last, the slots past ``count`` garbage bits.

    Row kinds cycle through: normal values at several spreads, heavy ties,
    one or more +inf at the head, all -inf, -inf after numbers, NaN tails,
    all NaN, empty, and spreads wide enough that exp(value / T) underflows.
    """
    rng = np.random.default_rng(seed)
    val = rng.integers(0, 1 << 16, size=(rows, k), dtype=np.uint16)
    count = np.empty(rows, np.int32)
    kinds = 10
    for r in range(rows):
        kind = r % kinds
        n = k if rng.random() < 0.6 else int(rng.integers(0, k + 1))
        sigma = float(rng.choice([0.05, 0.25, 1.0, 4.0, 16.0]))
        z = rng.standard_normal(n).astype(np.float32) * np.float32(sigma)
        if kind == 1:                                   # heavy ties
            z = rng.choice(np.float32([0.5, 0.0, -1.25]), size=n)
        elif kind == 8:                                 # underflowing tail
            z = rng.uniform(-300.0, 3.0, size=n).astype(np.float32)
        bits = round_to_bf16(z)
        if kind == 2 and n:                             # +inf at the head
            bits[: int(rng.integers(1, n + 1))] = BF16_POS_INF
        elif kind == 3:                                 # nothing but -inf
            bits[:] = BF16_NEG_INF
        elif kind == 4 and n:                           # -inf after some numbers
            bits[int(rng.integers(0, n)):] = BF16_NEG_INF
        nan_tail = 0
        if kind == 5 and n:
            nan_tail = int(rng.integers(1, n + 1))
        elif kind == 6:
            nan_tail = n
        elif kind == 7:
            n = 0
        body = bits[: n - nan_tail]
        order = np.argsort(-bf16_to_float(body), kind="stable")
        val[r, : n - nan_tail] = body[order]
        val[r, n - nan_tail: n] = _nan_bits(rng, nan_tail)
        count[r] = n
    return val, count


# ----------------------------------------------------------------------------- draft head inputs

@dataclass
class HeadInputs:
    """Inputs of the draft head that feeds the top-k: ``hidden`` [rows, dim]
    and ``weight`` [vocab, dim], both uint16 bf16 bit patterns, plus k."""
    name: str
    hidden: np.ndarray
    weight: np.ndarray
    k: int

    @property
    def rows(self) -> int:
        return self.hidden.shape[0]

    @property
    def dim(self) -> int:
        return self.hidden.shape[1]

    @property
    def vocab(self) -> int:
        return self.weight.shape[0]


def head_inputs(rows: int, dim: int, vocab: int, k: int, seed: int) -> HeadInputs:
    """Hidden states i/16 and weights j/64 with i, j uniform in -8..8.

    Every value is a small integer over a power of two, so each product is a
    multiple of 2^-10 and every partial sum of a dot product over dim <= 2^13
    stays below 2^14 in magnitude: such sums are exact in fp32 and fp64 in
    any order, and the bf16 logits they round to are unique.  Integers of at
    most four significant bits make the bf16 values exact.  Rounded to bf16,
    the logits collide often, so the top-k meets many ties.
    """
    rng = np.random.default_rng(seed)
    hidden = round_to_bf16(rng.integers(-8, 9, size=(rows, dim)).astype(np.float32) / np.float32(16))
    weight = np.empty((vocab, dim), np.uint16)
    step = max(1, (1 << 24) // max(dim, 1))
    for v0 in range(0, vocab, step):
        v1 = min(vocab, v0 + step)
        weight[v0:v1] = round_to_bf16(rng.integers(-8, 9, size=(v1 - v0, dim)).astype(np.float32) / np.float32(64))
    return HeadInputs(f"head_{rows}x{dim}x{vocab}_k{k}", hidden, weight, k)


def config_head_draft(seed: int = 5) -> HeadInputs:
    """The draft head of the pages' workload: 15 rows x 98592 columns, k = 16,
    from hidden states of 2048 dims (the pages do not give the drafter's width)."""
    return head_inputs(15, 2048, 98592, 16, seed)


def config_head_wide(seed: int = 6) -> HeadInputs:
    """The 16 x 248320, k = 64 shape as a head (2048 dims)."""
    return head_inputs(16, 2048, 248320, 64, seed)
