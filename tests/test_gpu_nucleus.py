"""GPU parity of tf_topk_nucleus_bf16, the nucleus (top-p) step over top-k
lists (the sampling settings of the TensorFold PR #3069 page, "Receipt":
temperature 0.7, top-k 20, top-p 0.95), against the float64 oracle.

Tolerance, from the kernel's fp32 arithmetic: x = (v - best) / T takes two
roundings (|dx| <= 2^-23 |x|), expf is within 2 ulp, a scan of at most 64
positive terms is within 63 * 2^-24 of its sum and the final division adds
2^-24.  With p |x| <= 1/e for every kept entry this bounds the error of a
probability by 2^-23 / e + 1e-5 * p: the test allows 1e-7 + 1e-5 * p.  The
cut (keep) is a float comparison of the running mass with top_p: the GPU's
cut must be one the float64 masses allow within DELTA = 2e-5 (the scan's error
bound, doubled); where it is, the probabilities are compared with the
oracle's renormalised at the GPU's cut."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from oracle.nucleus import nucleus, nucleus_row, values_of
from wide_bf16_row_gb300 import synth

pytestmark = pytest.mark.gpu

ATOL, RTOL, DELTA = 1e-7, 1e-5, 2e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from wide_bf16_row_gb300 import build
    build.build()


CODES = {"bf16": 0, "f16": 1, "f32": 2}


def _gpu(val: np.ndarray, count: np.ndarray, temperature: float, top_p: float, dtype: str = "bf16"):
    import torch

    from wide_bf16_row_gb300 import topk

    sint = np.int32 if dtype == "f32" else np.int16
    v = torch.from_numpy(np.ascontiguousarray(val).view(sint)).cuda()
    c = torch.from_numpy(np.ascontiguousarray(count, dtype=np.int32)).cuda()
    if dtype == "bf16":
        prob, keep = topk.nucleus_bf16(v, c, temperature, top_p)
    else:
        prob, keep = topk.nucleus(v, c, temperature, top_p, dtype=CODES[dtype])
    torch.cuda.synchronize()
    return prob.cpu().numpy(), keep.cpu().numpy()


def _check(val: np.ndarray, count: np.ndarray, temperature: float, top_p: float, what: str, dtype: str = "bf16"):
    prob, keep = _gpu(val, count, temperature, top_p, dtype)
    _compare(prob, keep, val, count, temperature, top_p, what, dtype)


def _compare(prob, keep, val, count, temperature: float, top_p: float, what: str, dtype: str = "bf16"):
    # the kernel sees the float32 values of T and top_p
    t32, p32 = float(np.float32(temperature)), float(np.float32(top_p))
    ref_prob, ref_keep, soft = nucleus(val, count, t32, p32, dtype=dtype)
    rows, k = val.shape
    assert prob.shape == (rows, k) and keep.shape == (rows,)
    moved = 0
    for r in range(rows):
        m, m_ref = int(keep[r]), int(ref_keep[r])
        exp = ref_prob[r]
        if m != m_ref:
            # only a cut the float64 masses put within DELTA of top_p may move
            cum = np.cumsum(soft[r])
            assert 1 <= m <= k and p32 < 1.0 and temperature > 0, f"{what} row {r}: keep {m} vs {m_ref}"
            assert cum[m - 1] >= p32 - DELTA and (m == 1 or cum[m - 2] < p32 + DELTA), \
                f"{what} row {r}: keep {m} is not a valid cut (oracle {m_ref})"
            n = max(0, min(k, int(count[r])))
            vals = [float(x) for x in values_of(val[r, :n], dtype)]
            exp = np.zeros(k)
            exp[:n] = nucleus_row(vals, t32, p32, keep=m)[2]
            moved += 1
        err = np.abs(prob[r] - exp)
        bad = err > ATOL + RTOL * exp
        assert not bad.any(), (f"{what} row {r}: prob {prob[r][bad][:4]} vs {exp[bad][:4]} "
                               f"(keep {m}, T {temperature}, top_p {top_p})")
    assert moved <= max(2, rows // 100), f"{what}: {moved} cuts moved"


@pytest.mark.parametrize("k", [1, 8, 20, 33, 64])
@pytest.mark.parametrize("temperature,top_p", [(0.7, 0.95), (0.7, 1.0), (0.0, 0.95), (0.3, 0.5),
                                               (1.0, 0.9), (5.0, 0.99), (1e-3, 0.95)])
def test_ranked_lists(k, temperature, top_p):
    val, count = synth.ranked_lists(600, k, seed=100 + k)
    _check(val, count, temperature, top_p, f"k{k}")


def test_exact_cuts_on_ties():
    """Equal values: every mass is a multiple of 1/n, exact in both precisions,
    so the cut is ceil(top_p * n) on both sides with no slack."""
    rows, k = 64, 16
    val = np.full((rows, k), synth.round_to_bf16(np.float32([1.5]))[0], dtype=np.uint16)
    count = np.array([1 + r % k for r in range(rows)], dtype=np.int32)
    for top_p in (0.25, 0.5, 0.75, 0.125):
        prob, keep = _gpu(val, count, 0.7, top_p)
        _, ref_keep, _ = nucleus(val, count, 0.7, top_p)
        assert np.array_equal(keep, ref_keep)
        for r in range(rows):
            assert np.allclose(prob[r, : keep[r]], 1.0 / keep[r], rtol=0, atol=1e-7)
            assert not prob[r, keep[r]:].any()


def test_after_the_top_k_on_the_draft_window():
    """The two steps queued back to back on 256 x 248320 (k = 20) with the
    receipt's settings; the expected lists come from the CPU top-k oracle."""
    import torch

    from tests.gpu_util import device_matrix
    from wide_bf16_row_gb300 import topk

    w = synth.config_draft_window()
    view, hold = device_matrix(w.logits, w.cols)
    idx, val, count, mask = topk.topk_bf16(view, w.k)
    prob, keep = topk.nucleus_bf16(val, count, 0.7, 0.95)
    torch.cuda.synchronize()
    ref = oracle.topk(w.logits, w.cols, w.k)
    assert np.array_equal(val.view(torch.int16).cpu().numpy().view(np.uint16), ref[1])
    assert np.array_equal(count.cpu().numpy(), ref[2])
    _compare(prob.cpu().numpy(), keep.cpu().numpy(), ref[1], ref[2], 0.7, 0.95, "draft window")
    del hold, idx, mask


def test_rows_beyond_one_block_and_counts_out_of_range():
    """More rows than one CTA's warps (a ragged last CTA); counts above k (on
    full lists) and below 0 are clamped to the list."""
    val, count = synth.ranked_lists(8 * 37 + 5, 20, seed=9)
    rows = np.arange(len(count))
    count[(count == 20) & (rows % 3 == 0)] = 25     # full lists: entries past k do not exist
    count[3::11] = -4
    _check(val, count, 0.7, 0.95, "clamped counts")


@pytest.mark.parametrize("dtype", ["f16", "f32"])
@pytest.mark.parametrize("temperature,top_p", [(0.7, 0.95), (0.0, 0.95), (1.0, 0.9), (5.0, 1.0)])
def test_other_formats(dtype, temperature, top_p):
    """The same ranked lists as fp16 (rounded) and fp32 (widened) values: the
    order survives (rounding is monotone), NaN and infinities map to the
    format's own."""
    val, count = synth.ranked_lists(600, 20, seed=321)
    vals = synth.bf16_to_float(val)
    with np.errstate(over="ignore", invalid="ignore"):
        bits = vals.astype(np.float16).view(np.uint16) if dtype == "f16" else np.ascontiguousarray(vals).view(np.uint32)
    _check(bits, count, temperature, top_p, f"{dtype} T{temperature} p{top_p}", dtype)
