"""Each plausible mistake in the nucleus (top-p) oracle fails at least one of
its pins.

A mutant is the oracle's source with one planted mistake (a text
substitution), loaded as a module of its own on the CPU; every pin of
tests/test_nucleus_pins.py is then run with the mutant's functions in place
of the oracle's.  A pin that raises -- an assertion or a crash -- has caught
it.
"""
from __future__ import annotations

import importlib.util
import types
from pathlib import Path

import pytest

from tests import test_nucleus_pins as pins

SOURCE = Path(__file__).resolve().parent.parent / "oracle" / "nucleus.py"

# name -> (text in the oracle, what the mutant has instead)
MUTANTS = {
    "temperature dropped": ("math.exp((v - top) / temperature)", "math.exp(v - top)"),
    "exponent sign flipped": ("math.exp((v - top) / temperature)", "math.exp((top - v) / temperature)"),
    "cut needs strictly more than top_p": ("if acc >= need:", "if acc > need:"),
    "kept prefix not renormalised": ("out = [x / kept for x in w[:keep]]", "out = [x / total for x in w[:keep]]"),
    "greedy spreads the mass": ("p = [1.0] + [0.0] * (n - 1)", "p = [1.0 / n] * n"),
    "infinite best shares with every entry": ("w = [1.0 if v == top else 0.0 for v in vals]",
                                              "w = [1.0 for v in vals]"),
    "NaN entries kept": ("n = next((i for i, v in enumerate(vals) if math.isnan(v)), size)", "n = size"),
    "top_p of one cuts the tail": ("elif top_p >= 1.0:", "elif top_p > 1.0:"),
    "fp16 lists decoded as bf16": ('if dtype == "f16":', 'if dtype == "f16 (never)":'),
    "fixed keep ignored": ("if keep is not None:", "if False:"),
    "negative count reads entries": ("n = max(0, min(k, int(count[r])))", "n = min(k, int(count[r]))"),
}

PIN_TESTS = [getattr(pins, name) for name in dir(pins) if name.startswith("test_")]


def _mutant(name: str) -> types.ModuleType:
    old, new = MUTANTS[name]
    text = SOURCE.read_text()
    assert text.count(old) == 1, f"the oracle no longer holds {old!r}"
    spec = importlib.util.spec_from_loader(f"nucleus_mutant_{abs(hash(name))}", loader=None)
    mod = importlib.util.module_from_spec(spec)
    exec(compile(text.replace(old, new), str(SOURCE), "exec"), mod.__dict__)
    return mod


def test_the_pins_pass_on_the_oracle_itself():
    for pin in PIN_TESTS:
        pin()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    bad = _mutant(name)
    for fn in ("nucleus", "nucleus_row", "values_of"):
        monkeypatch.setattr(pins, fn, getattr(bad, fn))
    caught = []
    for pin in PIN_TESTS:
        try:
            pin()
        except Exception:  # an assertion, or a crash the mistake causes
            caught.append(pin.__name__)
    assert caught, f"mutant '{name}' passed every pin"
