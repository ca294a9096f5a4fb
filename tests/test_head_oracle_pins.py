"""Pins of the draft-head oracle (oracle/head.py): the bf16 rounding against
torch's CPU conversion and hand-derived cases, the logits against exact
rational arithmetic with an independent rounding, and the top-k of tiny heads
against a plain sort.  The head's reading -- an LM head whose fp32 sum is
rounded to bf16, feeding the top-k of TensorFold PR #713, change 3 -- is
stated in the oracle's docstring; the planted mistakes at the end each fail
at least one pin."""
from __future__ import annotations

import importlib.util
import types
from fractions import Fraction
from pathlib import Path

import numpy as np
import pytest

import oracle
from oracle import head
from wide_bf16_row_gb300 import synth

SOURCE = Path(__file__).resolve().parent.parent / "oracle" / "head.py"


def _exact(bits: int) -> Fraction:
    """The exact value of finite bf16 bits, from sign, exponent and fraction."""
    s, e, f = bits >> 15, (bits >> 7) & 0xFF, bits & 0x7F
    mag = Fraction(f, 128) * Fraction(2) ** -126 if e == 0 else (1 + Fraction(f, 128)) * Fraction(2) ** (e - 127)
    return -mag if s else mag


def _nearest_bf16(x: Fraction) -> int:
    """bf16 bits nearest to a rational (ties to the even last bit), by search
    over the finite positive bf16 values; past the largest, infinity."""
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    lo, hi = 0, 0x7F7F                    # bits order like values for positives
    if a > _exact(0x7F7F):
        up = _exact(0x7F7F) + (_exact(0x7F7F) - _exact(0x7F7E)) / 2
        if a > up or (a == up):           # the halfway point rounds to the even one: infinity (0x7F80)
            return sign | 0x7F80
        return sign | 0x7F7F
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if _exact(mid) <= a:
            lo = mid
        else:
            hi = mid
    if _exact(lo) == a:
        return sign | lo
    d_lo, d_hi = a - _exact(lo), _exact(hi) - a
    pick = lo if d_lo < d_hi else hi if d_hi < d_lo else (lo if lo % 2 == 0 else hi)
    return sign | pick


# ----------------------------------------------------------------------------- rounding

def test_rounding_hand_cases():
    cases = {
        0x3F808000: 0x3F80,  # 1 + 2^-8: halfway, the even neighbour is 1.0
        0x3F818000: 0x3F82,  # halfway above an odd last bit: up
        0x3F808001: 0x3F81,  # just above half: up
        0x3F807FFF: 0x3F80,  # just below half: down
        0x7F7F8000: 0x7F80,  # halfway past the largest bf16: to infinity (even)
        0x7F7F7FFF: 0x7F7F,
        0xFF7F8000: 0xFF80,
        0x00008000: 0x0000,  # subnormal halfway to the even zero
        0x00018000: 0x0002,
        0x80008000: 0x8000,
        0x7F800000: 0x7F80,
        0xFF800000: 0xFF80,
    }
    x = np.array(list(cases), dtype=np.uint32).view(np.float32)
    assert head.round_f32_to_bf16(x).tolist() == list(cases.values())
    nan = np.array([0x7FC00001, 0xFF800001], dtype=np.uint32).view(np.float32)
    out = head.round_f32_to_bf16(nan)
    assert all((int(b) & 0x7FFF) > 0x7F80 for b in out)


def test_rounding_matches_torch_cpu():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    u = rng.integers(0, 1 << 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    u[:50_000] = (u[:50_000] & np.uint32(0xFFFF0000)) | np.uint32(0x8000)   # exact halves
    u[50_000:60_000] = (u[50_000:60_000] & np.uint32(0x807FFFFF)) | np.uint32(0x7F000000)  # near the top
    x = u.view(np.float32)
    finite = np.isfinite(x)
    ours = head.round_f32_to_bf16(x[finite])
    theirs = torch.from_numpy(x[finite].copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, theirs)


# ----------------------------------------------------------------------------- logits

def _tiny(rows, dim, vocab, seed):
    return synth.head_inputs(rows, dim, vocab, 1, seed)


@pytest.mark.parametrize("rows,dim,vocab,seed", [(1, 8, 5, 0), (3, 16, 11, 1), (4, 40, 9, 2), (2, 64, 7, 3)])
def test_logits_against_exact_rationals(rows, dim, vocab, seed):
    h = _tiny(rows, dim, vocab, seed)
    got = head.head_logits(h.hidden, h.weight)
    for r in range(rows):
        for v in range(vocab):
            s = sum(_exact(int(h.hidden[r, d])) * _exact(int(h.weight[v, d])) for d in range(dim))
            assert int(got[r, v]) == _nearest_bf16(s), (r, v)


def test_logits_on_scaled_inputs_and_exact_halves():
    # a sum landing exactly halfway between two bf16 values rounds to the even one
    hidden = synth.round_to_bf16(np.array([[1.0, 2.0 ** -8]], np.float32))      # 1 + 2^-8 after the product
    weight = synth.round_to_bf16(np.array([[1.0, 1.0], [1.0, 3.0]], np.float32))
    got = head.head_logits(hidden, weight)
    assert got.tolist() == [[0x3F80, 0x3F82]]      # 1 + 2^-8 -> 1.0; 1 + 3 * 2^-8 -> 1 + 2^-6 (halfway, even)


def test_refuses_sums_float64_could_round():
    hidden = synth.round_to_bf16(np.array([[2.0 ** 60, 2.0 ** -60]], np.float32))
    weight = synth.round_to_bf16(np.array([[1.0, 1.0]], np.float32))
    with pytest.raises(ValueError):
        head.head_logits(hidden, weight)


# ----------------------------------------------------------------------------- top-k

@pytest.mark.parametrize("rows,dim,vocab,k,seed", [(2, 16, 40, 5, 4), (3, 8, 64, 64, 5), (1, 24, 129, 9, 6)])
def test_topk_against_a_plain_sort(rows, dim, vocab, k, seed):
    h = synth.head_inputs(rows, dim, vocab, k, seed)
    idx, val, count, mask = head.topk(h.hidden, h.weight, k)
    logits = head.head_logits(h.hidden, h.weight)
    for r in range(rows):
        vals = [float(_exact(int(b))) for b in logits[r]]
        order = sorted(range(vocab), key=lambda c: (-vals[c], c))[:k]
        n = min(k, vocab)
        assert idx[r, :n].tolist() == order
        assert val[r, :n].tolist() == [int(logits[r, c]) for c in order]
        assert count[r] == n and mask[r] == 0
        assert idx[r, n:].tolist() == [-1] * (k - n)


def test_topk_is_the_topk_oracle_on_the_logits():
    h = synth.head_inputs(5, 72, 300, 12, 7)
    logits = head.head_logits(h.hidden, h.weight)
    for a, b in zip(head.topk(h.hidden, h.weight, 12), oracle.topk(logits, 300, 12)):
        np.testing.assert_array_equal(a, b)


# ----------------------------------------------------------------------------- planted mistakes

MUTANTS = {
    "truncation instead of rounding": ("up = (lo > 0x8000) | ((lo == 0x8000) & ((hi & 1) == 1))", "up = lo > 0xFFFF"),
    "ties away from zero": ("up = (lo > 0x8000) | ((lo == 0x8000) & ((hi & 1) == 1))", "up = lo >= 0x8000"),
    "ties to odd": ("up = (lo > 0x8000) | ((lo == 0x8000) & ((hi & 1) == 1))",
                    "up = (lo > 0x8000) | ((lo == 0x8000) & ((hi & 1) == 0))"),
    "last dim dropped": ("exact = h @ w.T ", "exact = h[:, :-1] @ w[:, :-1].T "),
    "vocab rows shifted": ("w = bf16_values(weight[v0: v0 + block])",
                           "w = bf16_values(np.roll(weight, 1, axis=0)[v0: v0 + block])"),
    "bf16 read as its low half": ("b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)",
                                  "b = np.asarray(bits, dtype=np.uint16).astype(np.uint32)"),
}

PINS = [test_rounding_hand_cases, test_rounding_matches_torch_cpu, test_logits_on_scaled_inputs_and_exact_halves,
        lambda: test_logits_against_exact_rationals(3, 16, 11, 1),
        lambda: test_topk_against_a_plain_sort(2, 16, 40, 5, 4)]


def _mutant(name: str) -> types.ModuleType:
    old, new = MUTANTS[name]
    text = SOURCE.read_text()
    assert text.count(old) == 1, f"the oracle no longer holds {old!r}"
    spec = importlib.util.spec_from_loader(f"head_mutant_{abs(hash(name))}", loader=None)
    mod = importlib.util.module_from_spec(spec)
    exec(compile(text.replace(old, new), str(SOURCE), "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    bad = _mutant(name)
    monkeypatch.setitem(globals(), "head", bad)
    caught = []
    for pin in PINS:
        try:
            pin()
        except Exception:  # an assertion, or a crash the mistake causes
            caught.append(pin)
    assert caught, f"mutant '{name}' passed every pin"
