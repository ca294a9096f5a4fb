"""Pins that hold the CPU oracle to the definition, independently of itself.

The definition (TensorFold PR #713, "perf(qwen27): ... top-k use more of the
GPU"): change 3 fixes the order -- score descending, lower token index first
on equal scores; the "Exactness" table fixes the outputs (entries, a count and
a non-finite mask per row) and the cases (ties, both zeros, NaN, infinities,
padded strides).  The conventions the pages leave open are the oracle's
readings: NaN never selected, +0 == -0, count = min(k, non-NaN columns), mask
bits NaN/+inf/-inf, empty slots (-1, 0x7FC0).

Every pin compares the oracle with something that is not the oracle: a
separately written brute force, numpy's stable argsort, Python's sorted(),
hand-derived fixtures (tests/golden/), or properties of the definition.  The
mutant test builds deliberately broken oracles and checks that each one fails
at least one pin.
"""
from __future__ import annotations

import itertools
import math
import struct

import numpy as np
import pytest

from oracle import Oracle
from tests import golden_io
from wide_bf16_row_gb300 import synth

EMPTY_IDX = -1
EMPTY_VAL = 0x7FC0


def decode(bits: int) -> float:
    """bf16 bits -> Python float, through struct (independent of the oracle's decode)."""
    return struct.unpack(">f", struct.pack(">I", (int(bits) & 0xFFFF) << 16))[0]


def brute_force_row(bits, k):
    """Repeated argmax: k times, take the best unused non-NaN column (strict > keeps
    the lowest column among equal scores)."""
    vals = [decode(b) for b in bits]
    used = set()
    picked = []
    for _ in range(k):
        best = None
        for c, v in enumerate(vals):
            if c in used or math.isnan(v):
                continue
            if best is None or v > vals[best]:
                best = c
        if best is None:
            break
        used.add(best)
        picked.append(best)
    mask = 0
    for v in vals:
        if math.isnan(v):
            mask |= 1
        elif v == math.inf:
            mask |= 2
        elif v == -math.inf:
            mask |= 4
    idx = picked + [EMPTY_IDX] * (k - len(picked))
    val = [int(bits[c]) for c in picked] + [EMPTY_VAL] * (k - len(picked))
    return idx, val, len(picked), mask


def check_against(oracle: Oracle, logits: np.ndarray, cols: int, k: int, expect, dtype: str = "bf16") -> None:
    idx, val, count, mask = oracle.topk(logits, cols, k, nthreads=2, dtype=dtype)
    e_idx, e_val, e_count, e_mask = expect
    np.testing.assert_array_equal(count, np.asarray(e_count, np.int32))
    np.testing.assert_array_equal(mask, np.asarray(e_mask, np.uint32))
    np.testing.assert_array_equal(idx, np.asarray(e_idx, np.int32))
    np.testing.assert_array_equal(val, np.asarray(e_val, np.uint32 if dtype == "f32" else np.uint16))


# --------------------------------------------------------------------------- pins

def pin_bruteforce_alphabet(oracle: Oracle) -> None:
    """Every row of length 1..3 over {-inf, -1, -min sub, -0, +0, +min sub, +1, +inf, NaN},
    k = 1..4, against the repeated-argmax brute force."""
    alpha = synth.special_alphabet()
    for length in (1, 2, 3):
        rows = np.array(list(itertools.product(alpha, repeat=length)), np.uint16)
        for k in (1, 2, 3, 4):
            exp = [brute_force_row(r, k) for r in rows]
            check_against(oracle, rows, length, k,
                          ([e[0] for e in exp], [e[1] for e in exp], [e[2] for e in exp],
                           [e[3] for e in exp]))


def pin_bruteforce_random(oracle: Oracle) -> None:
    """Random short rows with copies and specials (incl. padded strides) vs brute force."""
    rng = np.random.default_rng(11)
    for cols, stride, k in ((5, 5, 3), (9, 11, 4), (16, 16, 16), (33, 40, 7), (70, 70, 64)):
        x = synth.mixed_rows(6, cols, seed=int(rng.integers(1 << 30)), row_stride=stride,
                             special_frac=0.2, dup_frac=0.2)
        exp = [brute_force_row(r[:cols], k) for r in x]
        check_against(oracle, x, cols, k,
                      ([e[0] for e in exp], [e[1] for e in exp], [e[2] for e in exp],
                       [e[3] for e in exp]))


def pin_numpy_argsort(oracle: Oracle) -> None:
    """numpy's stable argsort of -value (NaN last, -0 == +0) truncated to count."""
    for seed, cols, k in ((1, 1000, 64), (2, 4099, 20), (3, 257, 1)):
        x = synth.mixed_rows(5, cols, seed=seed, special_frac=0.05, dup_frac=0.05)
        with np.errstate(invalid="ignore"):
            v = synth.bf16_to_float(x).astype(np.float64)
        e_idx = np.full((5, k), EMPTY_IDX, np.int32)
        e_val = np.full((5, k), EMPTY_VAL, np.uint16)
        e_count = np.zeros(5, np.int32)
        e_mask = np.zeros(5, np.uint32)
        for r in range(5):
            order = np.argsort(-v[r], kind="stable")
            n = min(k, int(np.count_nonzero(~np.isnan(v[r]))))
            e_idx[r, :n] = order[:n]
            e_val[r, :n] = x[r, order[:n]]
            e_count[r] = n
            e_mask[r] = (1 if np.isnan(v[r]).any() else 0) | (2 if (v[r] == np.inf).any() else 0) \
                | (4 if (v[r] == -np.inf).any() else 0)
        check_against(oracle, x, cols, k, (e_idx, e_val, e_count, e_mask))


def pin_full_sort(oracle: Oracle) -> None:
    """k = cols gives the full stable sort (Python sorted on (-value, column))."""
    x = synth.mixed_rows(4, 300, seed=5, special_frac=0.1, dup_frac=0.1)
    cols = k = 300
    idx, val, count, _ = oracle.topk(x, cols, k, nthreads=1)
    for r in range(4):
        vals = [decode(b) for b in x[r]]
        order = sorted((c for c in range(cols) if not math.isnan(vals[c])),
                       key=lambda c: (-vals[c], c))
        assert count[r] == len(order)
        assert list(idx[r, : len(order)]) == order
        assert all(i == EMPTY_IDX for i in idx[r, len(order):])


def pin_prefix(oracle: Oracle) -> None:
    """top-k(k1) is the first k1 entries of top-k(k2) for k1 < k2."""
    x = synth.mixed_rows(6, 2000, seed=7, special_frac=0.02, dup_frac=0.05)
    big = oracle.topk(x, 2000, 64, nthreads=2)
    for k1 in (1, 2, 8, 20, 63):
        small = oracle.topk(x, 2000, k1, nthreads=2)
        np.testing.assert_array_equal(small[0], big[0][:, :k1])
        np.testing.assert_array_equal(small[1], big[1][:, :k1])
        np.testing.assert_array_equal(small[2], np.minimum(big[2], k1))
        np.testing.assert_array_equal(small[3], big[3])


def pin_edge_rows(oracle: Oracle) -> None:
    """All-zero, all-NaN and all-equal rows; a padded stride equals the packed copy."""
    cols, k = 500, 64
    rng = np.random.default_rng(3)
    zeros = (rng.integers(0, 2, size=(1, cols), dtype=np.uint16) << np.uint16(15))
    idx, val, count, mask = oracle.topk(zeros, cols, k)
    assert list(idx[0]) == list(range(k)) and count[0] == k and mask[0] == 0
    np.testing.assert_array_equal(val[0], zeros[0, :k])
    nans = (np.uint16(0x7F80) | rng.integers(1, 0x80, size=(1, cols), dtype=np.uint16)
            | (rng.integers(0, 2, size=(1, cols), dtype=np.uint16) << np.uint16(15)))
    idx, val, count, mask = oracle.topk(nans, cols, k)
    assert count[0] == 0 and mask[0] == 1
    assert (idx == EMPTY_IDX).all() and (val == EMPTY_VAL).all()
    same = np.full((1, cols), 0xC0A0, np.uint16)  # -5.0 everywhere
    idx, val, count, mask = oracle.topk(same, cols, k)
    assert list(idx[0]) == list(range(k)) and (val == 0xC0A0).all() and mask[0] == 0
    packed = synth.mixed_rows(7, 777, seed=9, special_frac=0.05)
    padded = np.full((7, 800), 0x7F80, np.uint16)  # +inf in the padding
    padded[:, 777:] = rng.integers(0, 1 << 16, size=(7, 23), dtype=np.uint16)
    padded[:, :777] = packed
    a = oracle.topk(packed, 777, 33)
    b = oracle.topk(padded, 777, 33)
    for u, w in zip(a, b):
        np.testing.assert_array_equal(u, w)


def pin_golden(oracle: Oracle) -> None:
    """Hand-derived fixtures under tests/golden/ (bf16, fp16 and fp32)."""
    fixtures = golden_io.all_fixtures()
    assert len(fixtures) >= 5 and {fx["dtype"] for fx in fixtures} == {"bf16", "f16", "f32"}
    for fx in fixtures:
        check_against(oracle, fx["logits"], fx["cols"], fx["k"],
                      (fx["idx"], fx["val"], fx["count"], fx["mask"]), dtype=fx["dtype"])


def pin_invariants(oracle: Oracle) -> None:
    """Values non-increasing, equal values in increasing columns, and nothing left out
    beats the last entry (a bigger unselected score, or an equal one at a lower column,
    would contradict the order)."""
    x = synth.mixed_rows(8, 3000, seed=13, special_frac=0.03, dup_frac=0.1)
    for k in (1, 5, 64):
        idx, val, count, mask = oracle.topk(x, 3000, k)
        for r in range(8):
            n = int(count[r])
            sel = list(idx[r, :n])
            vals = [decode(x[r, c]) for c in sel]
            assert [int(x[r, c]) for c in sel] == [int(b) for b in val[r, :n]]
            for i in range(n - 1):
                assert vals[i] >= vals[i + 1]
                if vals[i] == vals[i + 1]:
                    assert sel[i] < sel[i + 1]
            chosen = set(sel)
            for c in range(3000):
                if c in chosen:
                    continue
                v = decode(x[r, c])
                if math.isnan(v):
                    continue
                assert n == k, "a non-NaN column was left out of a short list"
                assert v < vals[-1] or (v == vals[-1] and c > sel[-1])


# ---- fp16 and fp32: the same definition, values decoded by numpy's own types

EMPTY_BY_DTYPE = {"f16": 0x7E00, "f32": 0x7FC00000}


def numpy_values(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Bit patterns -> float64 through numpy's float16 / float32 (not the oracle's decode)."""
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns widen to NaN
        if dtype == "f16":
            return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)
        return np.asarray(bits, np.uint32).view(np.float32).astype(np.float64)


def reference_rows(x: np.ndarray, cols: int, k: int, dtype: str):
    """Per row: non-NaN columns in stable order of -value, truncated to k; mask
    and empty slots by the readings."""
    rows = x.shape[0]
    bits = np.uint32 if dtype == "f32" else np.uint16
    e_idx = np.full((rows, k), EMPTY_IDX, np.int32)
    e_val = np.full((rows, k), EMPTY_BY_DTYPE[dtype], bits)
    e_count = np.zeros(rows, np.int32)
    e_mask = np.zeros(rows, np.uint32)
    for r in range(rows):
        v = numpy_values(x[r, :cols], dtype)
        order = [c for c in np.argsort(-v, kind="stable") if not math.isnan(v[c])]
        n = min(k, len(order))
        e_idx[r, :n] = order[:n]
        e_val[r, :n] = x[r, order[:n]]
        e_count[r] = n
        e_mask[r] = (1 if np.isnan(v).any() else 0) | (2 if (v == np.inf).any() else 0) \
            | (4 if (v == -np.inf).any() else 0)
    return e_idx, e_val, e_count, e_mask


def brute_force_rows(x: np.ndarray, k: int, dtype: str):
    """Repeated argmax over numpy-decoded values (strict > keeps the lowest column)."""
    rows, cols = x.shape
    bits = np.uint32 if dtype == "f32" else np.uint16
    e_idx = np.full((rows, k), EMPTY_IDX, np.int32)
    e_val = np.full((rows, k), EMPTY_BY_DTYPE[dtype], bits)
    e_count = np.zeros(rows, np.int32)
    e_mask = np.zeros(rows, np.uint32)
    for r in range(rows):
        vals = [float(v) for v in numpy_values(x[r], dtype)]
        used, picked = set(), []
        for _ in range(k):
            best = None
            for c, v in enumerate(vals):
                if c not in used and not math.isnan(v) and (best is None or v > vals[best]):
                    best = c
            if best is None:
                break
            used.add(best)
            picked.append(best)
        e_idx[r, :len(picked)] = picked
        e_val[r, :len(picked)] = x[r, picked]
        e_count[r] = len(picked)
        e_mask[r] = sum(b for b, hit in ((1, any(math.isnan(v) for v in vals)), (2, math.inf in vals),
                                          (4, -math.inf in vals)) if hit)
    return e_idx, e_val, e_count, e_mask


def pin_f16_f32_alphabet(oracle: Oracle) -> None:
    """Every row of length 1..3 over each format's special alphabet, k = 1..4,
    against the repeated-argmax brute force."""
    for dtype, alpha in (("f16", synth.special_alphabet_f16()), ("f32", synth.special_alphabet_f32())):
        for length in (1, 2, 3):
            rows = np.array(list(itertools.product(alpha, repeat=length)), alpha.dtype)
            for k in (1, 2, 4):
                check_against(oracle, rows, length, k, brute_force_rows(rows, k, dtype), dtype=dtype)


def pin_f16_f32_argsort(oracle: Oracle) -> None:
    """Random mixed rows (subnormals, specials, copies, low-half near-ties,
    padded strides) against numpy's stable argsort of -value."""
    for dtype, gen in (("f16", synth.mixed_rows_f16), ("f32", synth.mixed_rows_f32)):
        for seed, cols, stride, k in ((1, 1000, 1000, 64), (2, 4099, 4160, 20), (3, 257, 260, 1),
                                      (4, 300, 300, 300)):
            x = gen(4, cols, seed=seed, row_stride=stride, special_frac=0.08, dup_frac=0.05)
            check_against(oracle, x, cols, k, reference_rows(x, cols, k, dtype), dtype=dtype)


def pin_masked_rows(oracle: Oracle) -> None:
    """-inf masks (random, dense, a padded vocabulary's tail, every column)
    with a few +inf in each format: -inf is a number that sorts last and sets
    mask bit 4 (+inf bit 2); numpy's stable argsort of -value decides."""
    for dtype in ("bf16", "f16", "f32"):
        for seed, (frac, tail, pinf, k) in enumerate(((0.1, 0, 0.0, 64), (0.9, 0, 0.01, 300),
                                                      (0.0, 700, 0.0, 1024), (1.0, 0, 0.0, 5))):
            x = synth.masked_rows(3, 1000, seed=seed, mask_frac=frac, tail=tail, plus_inf_frac=pinf,
                                  row_stride=1000 + seed, fmt=dtype)
            if dtype == "bf16":
                wide = (x.astype(np.uint32) << np.uint32(16)).astype(np.uint32)
                exp = reference_rows(wide, 1000, k, "f32")
                exp = (exp[0], (exp[1] >> np.uint32(16)).astype(np.uint16), exp[2], exp[3])
            else:
                exp = reference_rows(x, 1000, k, dtype)
            assert all(exp[3] & 4) and not any(exp[3] & 1)
            check_against(oracle, x, 1000, k, exp, dtype=dtype)


PINS = [pin_bruteforce_alphabet, pin_bruteforce_random, pin_numpy_argsort, pin_full_sort,
        pin_prefix, pin_edge_rows, pin_golden, pin_invariants, pin_f16_f32_alphabet, pin_f16_f32_argsort,
        pin_masked_rows]


@pytest.fixture(scope="module")
def oracle():
    return Oracle(0)


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin, oracle):
    pin(oracle)


MUTANTS = {
    1: "ascending order",
    2: "ties to the higher column",
    3: "NaN kept and ranked as +inf",
    4: "-0 ranked below +0",
    5: "last column never read",
    6: "infinity mask bits swapped",
    7: "count ignores NaN columns",
    8: "empty slots hold value bits 0",
    9: "row stride ignored",
    10: "fp16 subnormals read as normals",
    11: "fp32 read from its high half only",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=[MUTANTS[m] for m in sorted(MUTANTS)])
def test_pins_catch_mutant(mutant):
    """A planted mistake in the oracle (built on the CPU) must fail at least one pin."""
    bad = Oracle(mutant)
    caught = []
    for pin in PINS:
        try:
            pin(bad)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"


def test_oracle_threads_agree(oracle):
    """Splitting rows over threads does not change any output."""
    x = synth.mixed_rows(13, 1500, seed=21, special_frac=0.02)
    a = oracle.topk(x, 1500, 17, nthreads=1)
    b = oracle.topk(x, 1500, 17, nthreads=5)
    for u, w in zip(a, b):
        np.testing.assert_array_equal(u, w)


def test_oracle_rejects_bad_arguments(oracle):
    with pytest.raises(RuntimeError):
        oracle.topk(np.zeros((2, 4), np.uint16), 5, 1)  # cols > stride
    with pytest.raises(RuntimeError):
        oracle.topk(np.zeros((2, 4), np.uint16), 4, 0)  # k < 1
