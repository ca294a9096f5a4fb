"""CPU oracle for the draft head with the top-k in its epilogue -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this module; the product path never does.

Source: the pull request page "perf(qwen27): a drafted round overlaps its
cache commit with the next draft, and the drafter's attention and top-k use
more of the GPU" (TensorFold PR #713), change 3: the top-k runs over the
draft head's rows of bf16 logits (15 rows x 98592 columns there).  The page
gives the logits' shape and format, not how the head makes them; the reading
taken here is the usual LM head, a matrix product with a [vocab][dim] weight
whose fp32 sum is rounded to bf16:

    logit[r][v] = bf16_rne( fp32( sum_d hidden[r][d] * weight[v][d] ) )

followed by exactly the top-k of the pages (``oracle.topk``: score
descending, lower column first, NaN never selected, count and non-finite
mask per row).

The sum is computed exactly, in float64, and this module refuses inputs for
which float64 could round it: every bf16 value is an integer times a power of
two, so with all hidden values multiples of 2^-a bounded by H and all weights
multiples of 2^-b bounded by W, every partial sum is a multiple of 2^-(a+b)
bounded by dim * H * W, and the sum is exact when dim * H * W * 2^(a+b) <
2^53.  The exact sum is then rounded to fp32 and to bf16, each to nearest
with ties to even (numpy's float64 -> float32 conversion is IEEE round to
nearest even; the bf16 step is written out below).
"""
from __future__ import annotations

import numpy as np

import oracle as _topk


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact: a bf16 is the top half of a binary32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 values -> bf16 bits, rounding to nearest, ties to even.

    The bf16 value is the float32's top 16 bits when the dropped low half is
    below half an ulp; the next bf16 up when it is above; on an exact half,
    whichever of the two has an even last bit.  Carrying into the exponent is
    the correct result (up to +-inf past the largest bf16).  A NaN stays a
    NaN (quiet, sign kept)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    hi = (u >> np.uint32(16)).astype(np.uint32)
    lo = u & np.uint32(0xFFFF)
    up = (lo > 0x8000) | ((lo == 0x8000) & ((hi & 1) == 1))
    out = (hi + up.astype(np.uint32)) & np.uint32(0xFFFF)
    nan = (u & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    out = np.where(nan, (hi & np.uint32(0x8000)) | np.uint32(0x7FC0), out)
    return out.astype(np.uint16)


def _grain_and_bound(bits: np.ndarray) -> tuple[int, float]:
    """(a, M) over a bf16 array: every value is a multiple of 2^-a and
    |value| <= M.  Taken over the distinct bit patterns present."""
    present = np.flatnonzero(np.bincount(np.asarray(bits, dtype=np.uint16).ravel(), minlength=1 << 16))
    v = bf16_values(present.astype(np.uint16))
    nz = v[v != 0]
    if nz.size == 0:
        return 0, 0.0
    m, e = np.frexp(np.abs(nz))          # |v| = m * 2^e with m in [0.5, 1): m * 256 is an integer
    sig = np.rint(m * 256).astype(np.int64)
    tz = np.zeros_like(sig)
    while np.any((sig & 1) == 0):        # strip the significand's trailing zero bits
        even = (sig & 1) == 0
        tz[even] += 1
        sig[even] >>= 1
    a = int(np.max(-(e.astype(np.int64) - 8 + tz)))
    return a, float(np.max(np.abs(nz)))


def head_logits(hidden: np.ndarray, weight: np.ndarray, block: int = 16384) -> np.ndarray:
    """[rows][dim] and [vocab][dim] bf16 bits -> [rows][vocab] bf16 logit bits."""
    hidden = np.asarray(hidden, dtype=np.uint16)
    weight = np.asarray(weight, dtype=np.uint16)
    h = bf16_values(hidden)
    if not np.isfinite(h).all() or np.any((weight & 0x7F80) == 0x7F80):
        raise ValueError("the head oracle takes finite inputs")
    dim = hidden.shape[1]
    a, hb = _grain_and_bound(hidden)
    b, wb = _grain_and_bound(weight)
    if dim * hb * wb * 2.0 ** (a + b) >= 2.0 ** 53:
        raise ValueError("float64 could round this sum; the oracle refuses such inputs")
    vocab = weight.shape[0]
    out = np.empty((hidden.shape[0], vocab), np.uint16)
    for v0 in range(0, vocab, block):
        w = bf16_values(weight[v0: v0 + block])
        exact = h @ w.T                              # exact: see the module docstring
        out[:, v0: v0 + block] = round_f32_to_bf16(exact.astype(np.float32))
    return out


def topk(hidden: np.ndarray, weight: np.ndarray, k: int):
    """(idx, val bits, count, mask) of every row of the head's logits, as
    ``oracle.topk`` gives them for a [rows][vocab] bf16 matrix."""
    logits = head_logits(hidden, weight)
    return _topk.topk(logits, logits.shape[1], k)
