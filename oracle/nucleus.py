"""CPU oracle for the nucleus (top-p) step after the top-k -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` may import this module; the product path never does.

Source: the pull request page "qwen27 metal: restore the long-copy driver for
a lone greedy stream on M5 (#3013) - #3069" (TensorFold), section "Receipt":
drafted streams are sampled at temperature 0.7 with top-k 20 and top-p 0.95.
The pages name the settings but not the procedure; the reading taken here is
the usual one, top-k first and then top-p:

  * a row's candidates are its top-k entries (best first, ``count`` of them);
  * at temperature T > 0 their probabilities are the softmax of value / T over
    those entries alone;
  * the kept prefix is the shortest one whose probabilities sum to at least
    top_p (at least one entry); top_p == 1 keeps every entry;
  * the kept entries' probabilities are renormalised to sum to 1, the others
    are 0;
  * T == 0 is greedy: the first entry alone, probability 1;
  * an infinite best value (+inf, or -inf when every entry is -inf) gives the
    entries equal to it equal shares and every other entry 0;
  * NaN is not a score: the top-k ranks it below every number, so NaN entries
    form the tail of a row and take no probability; a row of NaN alone keeps
    nothing (keep 0, all probabilities 0).

Everything is computed in float64 with a plain sequential sum.
"""
from __future__ import annotations

import math

import numpy as np


def nucleus_row(vals: list[float], temperature: float, top_p: float,
                keep: int | None = None) -> tuple[list[float], int, list[float]]:
    """One row: (probabilities of every entry, kept count, renormalised kept
    probabilities padded with zeros).  ``keep``, when given, fixes the kept
    count in place of the top-p cut (a caller comparing a result whose cut
    fell on the other side of a rounding boundary)."""
    size = len(vals)
    n = next((i for i, v in enumerate(vals) if math.isnan(v)), size)
    if n < size:
        p, keep, out = nucleus_row(vals[:n], temperature, top_p, keep)
        pad = [0.0] * (size - n)
        return p + pad, keep, out + pad
    if n == 0:
        return [], 0, []
    if temperature == 0.0:
        p = [1.0] + [0.0] * (n - 1)
        return p, 1, list(p)
    # unnormalised weights w: the probabilities are w / sum(w)
    top = vals[0]
    if math.isinf(top):
        w = [1.0 if v == top else 0.0 for v in vals]
    else:
        w = [math.exp((v - top) / temperature) for v in vals]
    total = 0.0
    for x in w:
        total += x
    p = [x / total for x in w]
    # the cut: the shortest prefix whose probabilities reach top_p, i.e. whose
    # weights reach top_p * total (compared on the weights, so a prefix that
    # reaches top_p exactly -- equal shares -- is decided without the
    # rounding of the division)
    if keep is not None:
        keep = max(0, min(int(keep), n))
    elif top_p >= 1.0:
        keep = n
    else:
        keep, acc, need = n, 0.0, top_p * total
        for i, x in enumerate(w):
            acc += x
            if acc >= need:
                keep = i + 1
                break
    kept = 0.0
    for x in w[:keep]:
        kept += x
    out = [x / kept for x in w[:keep]] + [0.0] * (n - keep) if keep else [0.0] * n
    return p, keep, out


def values_of(bits: np.ndarray, dtype: str = "bf16") -> np.ndarray:
    """Bit patterns of bf16, fp16 or fp32 values -> float64 (exact)."""
    b = np.asarray(bits)
    with np.errstate(invalid="ignore"):
        if dtype == "f16":
            return b.astype(np.uint16).view(np.float16).astype(np.float64)
        if dtype == "f32":
            return b.astype(np.uint32).view(np.float32).astype(np.float64)
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def nucleus(val_bits: np.ndarray, count: np.ndarray, temperature: float, top_p: float, dtype: str = "bf16"):
    """Rows of top-k results -> (prob float64 [rows][k], keep int [rows], and
    the pre-truncation softmax float64 [rows][k]).  ``val_bits`` holds bit
    patterns of ``dtype`` ("bf16", "f16" or "f32")."""
    rows, k = val_bits.shape
    values = values_of(val_bits, dtype)
    prob = np.zeros((rows, k))
    soft = np.zeros((rows, k))
    keep = np.zeros(rows, dtype=np.int64)
    for r in range(rows):
        n = max(0, min(k, int(count[r])))     # a list holds at most k entries
        vals = [float(v) for v in values[r, :n]]
        p, m, out = nucleus_row(vals, temperature, top_p)
        soft[r, :n] = p
        prob[r, :n] = out
        keep[r] = m
    return prob, keep, soft
