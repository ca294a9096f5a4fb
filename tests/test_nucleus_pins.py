"""Pins of the nucleus (top-p) oracle against closed forms and invariants
(the sampling settings of the TensorFold PR #3069 page, "Receipt": temperature
0.7, top-k 20, top-p 0.95; the procedure is the usual top-k-then-top-p
reading stated in oracle/nucleus.py)."""
from __future__ import annotations

import math

import numpy as np
import pytest

from oracle.nucleus import nucleus, nucleus_row, values_of


def test_two_values_follow_the_logistic_closed_form():
    # p0 = 1 / (1 + e^{-(a - b)/T}): a dropped temperature or a flipped sign fails
    for a, b, t in ((3.0, 1.0, 0.7), (0.5, -2.25, 2.0), (10.0, 9.5, 0.1)):
        p, keep, _ = nucleus_row([a, b], t, 1.0)
        assert p[0] == pytest.approx(1.0 / (1.0 + math.exp(-(a - b) / t)), rel=1e-12)
        assert p[1] == pytest.approx(1.0 - p[0], rel=1e-12, abs=1e-15)
        assert keep == 2


def test_equal_values_share_equally_and_keep_the_ceiling():
    # (4, 0.5): the prefix of two reaches 0.5 exactly, and reaching it is enough
    for n, top_p, expect in ((4, 0.55, 3), (5, 0.15, 1), (8, 0.9, 8), (3, 0.4, 2), (4, 0.5, 2)):
        p, keep, out = nucleus_row([1.5] * n, 0.7, top_p)
        assert all(x == pytest.approx(1.0 / n) for x in p)
        assert keep == expect == math.ceil(top_p * n - 1e-12)
        assert sum(out) == pytest.approx(1.0)
        assert all(x == pytest.approx(1.0 / expect) for x in out[:expect])


def test_temperature_limits():
    vals = [4.0, 3.0, 1.0, -2.0]
    p, _, _ = nucleus_row(vals, 1e7, 1.0)          # very hot: uniform
    assert all(x == pytest.approx(0.25, abs=1e-6) for x in p)
    p, keep, _ = nucleus_row(vals, 1e-3, 0.95)      # very cold: the best alone
    assert p[0] == pytest.approx(1.0) and keep == 1
    p, keep, out = nucleus_row(vals, 0.0, 0.5)       # greedy
    assert (p, keep, out) == ([1.0, 0.0, 0.0, 0.0], 1, [1.0, 0.0, 0.0, 0.0])


def test_infinities():
    p, keep, out = nucleus_row([math.inf, math.inf, 5.0], 0.7, 0.9)
    assert p == [0.5, 0.5, 0.0] and keep == 2 and out == [0.5, 0.5, 0.0]
    p, keep, _ = nucleus_row([1.0, -math.inf], 0.7, 0.5)
    assert p == [1.0, 0.0] and keep == 1
    p, keep, _ = nucleus_row([-math.inf] * 3, 0.7, 0.5)
    assert p == pytest.approx([1 / 3] * 3) and keep == 2


def test_top_p_one_keeps_everything_and_empty_rows_keep_nothing():
    _, keep, out = nucleus_row([3.0, -1.0, -math.inf], 0.7, 1.0)
    assert keep == 3 and sum(out) == pytest.approx(1.0)
    assert nucleus_row([], 0.7, 0.9) == ([], 0, [])


def test_invariants_on_random_sorted_rows():
    rng = np.random.default_rng(7)
    for _ in range(200):
        n = int(rng.integers(1, 65))
        vals = sorted((rng.standard_normal(n) * 4).tolist(), reverse=True)
        t = float(rng.choice([0.3, 0.7, 1.0, 2.5]))
        top_p = float(rng.uniform(0.05, 0.999))
        p, keep, out = nucleus_row(vals, t, top_p)
        assert all(p[i] >= p[i + 1] for i in range(n - 1))             # sorted values, sorted mass
        cum = np.cumsum(p)
        assert cum[keep - 1] >= top_p and (keep == 1 or cum[keep - 2] < top_p)  # shortest prefix
        assert sum(out) == pytest.approx(1.0) and all(x == 0.0 for x in out[keep:])


def test_rows_entry_point_reads_counts():
    bits = np.array([[0x4040, 0x3F80, 0x0000], [0x7F80, 0x4000, 0x0000]], dtype=np.uint16)  # 3,1 | inf,2
    prob, keep, soft = nucleus(bits, np.array([2, 1]), 1.0, 0.99)
    assert keep.tolist() == [2, 1]
    assert soft[0, 0] == pytest.approx(1 / (1 + math.exp(-2.0)))
    assert prob[1].tolist() == [1.0, 0.0, 0.0] and prob[0, 2] == 0.0


def test_rows_entry_point_keeps_the_untruncated_softmax():
    bits = np.array([[0x3F80, 0x3F80, 0x3F80, 0x3F80]], dtype=np.uint16)  # four 1.0
    prob, keep, soft = nucleus(bits, np.array([4]), 0.7, 0.5)
    assert keep.tolist() == [2]
    assert soft[0].tolist() == [0.25] * 4 and prob[0].tolist() == [0.5, 0.5, 0.0, 0.0]


def test_nan_entries_take_no_probability():
    nan = math.nan
    p, keep, out = nucleus_row([2.0, 2.0, nan], 0.7, 0.9)
    assert p == [0.5, 0.5, 0.0] and keep == 2 and out == [0.5, 0.5, 0.0]
    assert nucleus_row([nan, nan], 0.7, 0.9) == ([0.0, 0.0], 0, [0.0, 0.0])
    assert nucleus_row([nan], 0.0, 0.9) == ([0.0], 0, [0.0])


def test_a_fixed_keep_replaces_the_cut():
    p, keep, out = nucleus_row([1.0, 1.0, 1.0, 1.0], 0.7, 0.3, keep=3)
    assert keep == 3 and out == pytest.approx([1 / 3, 1 / 3, 1 / 3, 0.0])
    for top_p in (0.2, 0.6, 0.97):   # fixing the cut the rule would take changes nothing
        vals = [2.5, 1.0, 0.25, -3.0]
        ref = nucleus_row(vals, 0.7, top_p)
        assert nucleus_row(vals, 0.7, 0.5, keep=ref[1]) == ref


def test_other_formats_decode_exactly():
    """fp16 and fp32 lists: the same steps on exactly decoded values."""
    assert values_of(np.array([0x3C00, 0x0001, 0xFC00], np.uint16), "f16").tolist() == [1.0, 2.0 ** -24, -math.inf]
    assert values_of(np.array([0x3F800001], np.uint32), "f32")[0] == 1.0 + 2.0 ** -23
    assert values_of(np.array([0x4040], np.uint16))[0] == 3.0
    f32 = np.array([[0x40400000, 0x3F800000, 0]], np.uint32)        # 3, 1
    prob, keep, soft = nucleus(f32, np.array([2]), 1.0, 0.99, dtype="f32")
    assert soft[0, 0] == pytest.approx(1 / (1 + math.exp(-2.0))) and keep.tolist() == [2]
    f16 = np.array([[0x3C00, 0x3C00, 0x3C00, 0x7E00]], np.uint16)    # 1, 1, 1, NaN
    prob, keep, soft = nucleus(f16, np.array([4]), 0.7, 0.5, dtype="f16")
    assert keep.tolist() == [2] and soft[0].tolist() == pytest.approx([1 / 3, 1 / 3, 1 / 3, 0.0])


def test_counts_outside_the_list_are_clamped():
    """A list holds k entries: a count above k reads k of them, a negative one none."""
    bits = np.array([[0x4040, 0x3F80, 0x3F80]], dtype=np.uint16)           # 3, 1, 1
    ref = nucleus(bits, np.array([3]), 0.7, 0.9)
    over = nucleus(bits, np.array([7]), 0.7, 0.9)
    for a, b in zip(ref, over):
        np.testing.assert_array_equal(a, b)
    prob, keep, soft = nucleus(bits, np.array([-2]), 0.7, 0.9)
    assert keep.tolist() == [0] and not prob.any() and not soft.any()
