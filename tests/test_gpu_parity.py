"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, bit
for bit, on seeded inputs -- every named workload at full size, the width x
rows x k sweep, an edge grid around warp/vector/chunk/span boundaries with
misaligned bases and padded strides, heavy-tie and NaN-heavy rows, and every
launch plan (the single-CTA control and 2/4/8/16-span clusters) against each
other.  Byte equality is the bar, as in the "Exactness" table of TensorFold
PR #713 ("perf(qwen27): ... top-k use more of the GPU")."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_same, gpu_topk
from wide_bf16_row_gb300 import synth

pytestmark = pytest.mark.gpu

# every launch plan: single-CTA control, 2/4/8/16-span clusters, persistent stream
ALL_PLANS = (1, 2, 4, 8, 16, 32)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from wide_bf16_row_gb300 import build
    build.build()


@pytest.mark.parametrize("name", sorted(synth.NAMED))
def test_named_workload_full_size(name):
    w = synth.NAMED[name]()
    exp = oracle.topk(w.logits, w.cols, w.k)
    assert_same(gpu_topk(w.logits, w.cols, w.k), exp, name)


@pytest.mark.parametrize("name", ["1x4096_k8", "15x98592_k16", "16x248320_k64_specials"])
@pytest.mark.parametrize("plan", ALL_PLANS)
def test_named_workload_every_plan(name, plan):
    w = synth.NAMED[name]()
    exp = oracle.topk(w.logits, w.cols, w.k)
    assert_same(gpu_topk(w.logits, w.cols, w.k, plan=plan), exp, f"{name} plan={plan}")


@pytest.mark.parametrize("width", synth.SWEEP_WIDTHS)
@pytest.mark.parametrize("rows", synth.SWEEP_ROWS)
def test_sweep(width, rows):
    for k in synth.SWEEP_KS:
        w = synth.config_sweep(width, rows, k)
        exp = oracle.topk(w.logits, w.cols, w.k)
        assert_same(gpu_topk(w.logits, w.cols, w.k), exp, w.name)


EDGE_COLS = (1, 2, 7, 8, 9, 31, 33, 63, 64, 65, 255, 257, 1000, 2047, 2049, 4095, 4096, 4097,
             16383, 16384, 16385, 16391, 32776, 65537, 98592, 262147, 300001)


@pytest.mark.parametrize("cols", EDGE_COLS)
def test_edge_grid(cols):
    rng = np.random.default_rng(cols)
    for stride_extra, offset in ((0, 0), (1, 3), (5, 1), (8, 7)):
        stride = cols + stride_extra
        x = synth.mixed_rows(3, cols, seed=int(rng.integers(1 << 30)), row_stride=stride,
                             special_frac=0.01, dup_frac=0.02)
        for k in (1, 2, 63, 64):
            exp = oracle.topk(x, cols, k)
            for plan in (0, 1, 16, 32):
                got = gpu_topk(x, cols, k, plan=plan, offset=offset)
                assert_same(got, exp, f"cols={cols} stride={stride} off={offset} k={k} plan={plan}")


def _tie_rows(cols: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    rows = []
    rows.append(rng.integers(0, 2, size=cols, dtype=np.uint16) << np.uint16(15))  # all +-0
    rows.append(np.full(cols, 0x3F80, np.uint16))                                   # all 1.0
    two = np.where(rng.random(cols) < 0.5, 0x4000, 0x3F80).astype(np.uint16)        # 2.0 / 1.0
    rows.append(two)
    top = synth.round_to_bf16(rng.standard_normal(cols).astype(np.float32))        # 600 tied maxima
    top[rng.choice(cols, size=min(cols, 600), replace=False)] = 0x4300              # 128.0
    rows.append(top)
    sparse = np.full(cols, 0xFF80, np.uint16)                                        # -inf with few finite
    sparse[rng.choice(cols, size=min(cols, 40), replace=False)] = 0x3F80
    rows.append(sparse)
    mostly_nan = np.full(cols, 0x7FC1, np.uint16)                                    # NaN with 10 zeros
    mostly_nan[rng.choice(cols, size=min(cols, 10), replace=False)] = 0x8000
    rows.append(mostly_nan)
    rows.append(np.full(cols, 0xFFC1, np.uint16))                                    # all -NaN
    asc = np.sort(synth.bf16_to_float(synth.round_to_bf16(                          # ascending: every
        rng.standard_normal(cols).astype(np.float32))))                              # chunk beats the last
    rows.append(synth.round_to_bf16(asc))
    rows.append(synth.round_to_bf16(asc[::-1].copy()))                               # descending
    return np.stack(rows)


@pytest.mark.parametrize("cols", (100, 5000, 16384, 40000, 98592, 248320))
@pytest.mark.parametrize("k", (1, 20, 64))
def test_heavy_ties_and_nan(cols, k):
    x = _tie_rows(cols, seed=cols + k)
    exp = oracle.topk(x, cols, k)
    for plan in ALL_PLANS:
        assert_same(gpu_topk(x, cols, k, plan=plan), exp, f"ties cols={cols} k={k} plan={plan}")


MASKS = ((0.1, 0, 0.0), (0.6, 0, 0.0), (0.0, 1000, 0.0), (0.1, 64, 0.0005))


@pytest.mark.parametrize("rows,cols,k", [(256, 248320, 20), (16, 248320, 64), (15, 98592, 16), (1024, 4096, 8)])
def test_masked_rows(rows, cols, k):
    """-inf masks (random, dense, a padded vocabulary's tail) with a few +inf:
    chunks whose only non-finite values are infinities keep their keys and
    only record the flags."""
    for i, (frac, tail, pinf) in enumerate(MASKS):
        x = synth.masked_rows(rows, cols, seed=cols + i, mask_frac=frac, tail=tail, plus_inf_frac=pinf,
                              row_stride=cols + (8 if i % 2 else 0))
        exp = oracle.topk(x, cols, k)
        for plan in (0, 1, 2, 8, 32):
            assert_same(gpu_topk(x, cols, k, plan=plan, offset=i), exp,
                        f"masked {rows}x{cols} k={k} mask={frac} tail={tail} +inf={pinf} plan={plan}")


def test_masked_rows_f16():
    from tests.test_gpu_wide import gpu_select

    for i, (frac, tail, pinf) in enumerate(MASKS):
        x = synth.masked_rows(24, 98592, seed=7 + i, mask_frac=frac, tail=tail, plus_inf_frac=pinf, fmt="f16")
        exp = oracle.topk(x, 98592, 16, dtype="f16")
        for plan in (0, 1, 8):
            assert_same(gpu_select(x, 98592, 16, "f16", plan=plan), exp, f"f16 masked mask={frac} plan={plan}")


def test_every_plan_agrees_on_random_rows():
    x = synth.mixed_rows(40, 70000, seed=99, row_stride=70003, special_frac=0.002, dup_frac=0.01)
    exp = oracle.topk(x, 70000, 37)
    for plan in (0,) + ALL_PLANS:
        for offset in (0, 5):
            assert_same(gpu_topk(x, 70000, 37, plan=plan, offset=offset), exp,
                        f"plan={plan} off={offset}")


def test_repeated_calls_and_streams_are_deterministic():
    import torch

    from tests.gpu_util import device_matrix, to_numpy
    from wide_bf16_row_gb300 import topk

    w = synth.config_draft_head()
    view, keep = device_matrix(w.logits, w.cols)
    first = to_numpy(topk.topk_bf16(view, w.k))
    streams = [torch.cuda.Stream() for _ in range(3)]
    outs = []
    for i in range(30):
        s = streams[i % 3]
        with torch.cuda.stream(s):
            outs.append(topk.topk_bf16(view, w.k, stream=s))
    torch.cuda.synchronize()
    for o in outs:
        assert_same(to_numpy(o), first, "repeat")
    del keep


def test_binding_accepts_bfloat16_and_one_row():
    import torch

    from tests.gpu_util import to_numpy
    from wide_bf16_row_gb300 import topk

    x = synth.config_draft_single()
    t = torch.from_numpy(x.logits.view(np.int16)).cuda().view(torch.bfloat16)
    exp = oracle.topk(x.logits, x.cols, x.k)
    assert_same(to_numpy(topk.topk_bf16(t, x.k)), exp, "bf16 2-D")
    assert_same(to_numpy(topk.topk_bf16(t[0], x.k)), exp, "bf16 1-D")
    # values come back as bf16 numbers equal to the selected logits
    idx, val, _, _ = topk.topk_bf16(t, x.k)
    assert torch.equal(val[0], t[0, idx[0].long()])


def test_gpu_guard_errors_leave_outputs_untouched():
    import torch

    from wide_bf16_row_gb300 import topk

    x = torch.zeros((4, 100), dtype=torch.int16, device="cuda")
    idx = torch.full((4, 8), 1234, dtype=torch.int32, device="cuda")
    val = torch.full((4, 8), 77, dtype=torch.int16, device="cuda")
    cnt = torch.full((4,), 5, dtype=torch.int32, device="cuda")
    msk = torch.full((4,), 9, dtype=torch.int32, device="cuda")
    st = topk.tf_topk_bf16_with_plan(x.data_ptr(), 4, 100, 100, 8, idx.data_ptr(), val.data_ptr(),
                                     cnt.data_ptr(), msk.data_ptr(), 3, None)
    assert st == topk.ERR_PLAN
    st = topk.tf_topk_bf16(x.data_ptr(), 4, 100, 100, 65, idx.data_ptr(), val.data_ptr(),
                           cnt.data_ptr(), msk.data_ptr(), None)
    assert st == topk.ERR_K
    torch.cuda.synchronize()
    assert (idx == 1234).all() and (val == 77).all() and (cnt == 5).all() and (msk == 9).all()
    with pytest.raises(topk.TopkError):
        topk.topk_bf16(x, 0)


def test_plan_table():
    """AUTO's choice follows the documented rule (4 cluster-kernel CTAs an SM,
    16384-column chunks): with a row per SM or more, one CTA per row (SINGLE)
    for rows of at most one chunk or when two spans a row would take three
    waves or more, else CLUSTER2; with fewer rows, the span count that brings
    the grid to about two CTAs per SM without spans under half a chunk (a
    chunk for k > 32), down to one."""
    import torch

    from wide_bf16_row_gb300 import topk

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    chunk = 16384

    def rule(rows, cols, k):
        if rows >= sms:
            return 1 if (cols <= chunk or 2 * rows >= 3 * 4 * sms) else 2
        s = 2
        while s < 16 and rows * s < 2 * sms:
            s *= 2
        while s > 1 and cols // s < (chunk if k > 32 else chunk // 2):
            s //= 2
        return s

    for rows, cols in ((1, 100), (1, 4096), (15, 98592), (16, 248320), (256, 248320), (1024, 248320),
                       (1024, 4096), (512, 8192), (640, 248320), (sms, chunk), (sms, chunk + 1), (4, 98592)):
        for k in (8, 20, 64):
            got = topk.plan(rows, cols, k)
            assert got in ALL_PLANS and got == rule(rows, cols, k), (rows, cols, k, got)
    assert topk.plan(256, 248320, 20) == 2 and topk.plan(15, 98592, 16) == 8
    assert topk.device_fault() == 0
