"""Host-side pieces of the benchmark, on CPU: the reference arm's JSON line
(the oracle timed on the host cores), the formats the --dtype lines feed the
kernels, and the run labels that name their profiles."""
from __future__ import annotations

import io
import json
from contextlib import redirect_stdout

import numpy as np

import bench
from wide_bf16_row_gb300 import synth


def _line(argv) -> dict:
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(argv)
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1, lines
    return json.loads(lines[0])


def test_reference_arm_prints_one_contract_line():
    d = _line(["--impl", "reference", "--steps", "6", "--warmup", "3", "--workload", "1x4096_k8"])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "rows/s" and d["value"] > 0
    assert d["steps"] == 6 and d["gpu_launches"] == 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "1x4096_k8" and "format" not in d["config"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_format_and_k():
    d = _line(["--impl", "reference", "--steps", "4", "--warmup", "3", "--workload", "1x4096_k8",
               "--dtype", "f32", "--k", "100"])
    assert d["config"]["workload"] == "1x4096_k100_f32"
    assert d["config"]["format"] == "f32" and d["config"]["k"] == 100


def test_warmup_below_three_is_refused():
    import pytest
    with pytest.raises(SystemExit):
        bench.main(["--impl", "reference", "--steps", "4", "--warmup", "2"])


def test_format_bits_keep_the_values():
    w = synth.config_draft_single()
    f32 = bench.format_bits(w, "f32")
    assert f32.dtype == np.uint32
    # fp32 widening is exact: every value equals its bf16 original
    np.testing.assert_array_equal(f32.view(np.float32), synth.bf16_to_float(w.logits))
    f16 = bench.format_bits(w, "f16")
    assert f16.dtype == np.uint16
    vals = synth.bf16_to_float(w.logits).astype(np.float64)
    got = f16.view(np.float16).astype(np.float64)
    # round to nearest: within half an fp16 step of the original (N(0,1) values: no overflow)
    assert np.all(np.abs(got - vals) <= np.abs(vals) * 2.0 ** -11 + 2.0 ** -25)
    assert bench.format_bits(w, "bf16") is w.logits


def test_run_labels():
    w = synth.config_draft_window()
    assert bench.run_label(w, "bf16", 20) == "256x248320_k20"
    assert bench.run_label(w, "f16", 20) == "256x248320_k20_f16"
    assert bench.run_label(w, "bf16", 1024) == "256x248320_k1024_bf16"
