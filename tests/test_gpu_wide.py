"""GPU parity of tf_topk_select -- bf16, fp16 and fp32 rows, k up to 1024 --
against the CPU oracle, byte for byte (the order of TensorFold PR #713,
change 3, and the "Exactness" table's count and mask, applied to the two
further formats and to larger k).

Cases: every format over k from 1 to 1024; padded strides and row bases off
the 16-byte grid (the unaligned head and tail); rows shorter than k; the
heavy-tie fallback (all +-0, few distinct values, a k-th key shared by
thousands of columns); all-NaN rows; fp32 near-ties in the low half; the
256 x 248320 bench shape forced through the wide kernel; bf16 with k <= 64
through tf_topk_select against tf_topk_bf16; and fp16 with k <= 64 on the
cluster plans it shares with bf16 (the same key map, fp16's special
values)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from wide_bf16_row_gb300 import synth

pytestmark = pytest.mark.gpu

CODES = {"bf16": 0, "f16": 1, "f32": 2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from wide_bf16_row_gb300 import build
    build.build()


def _device(x: np.ndarray, cols: int, offset: int = 0):
    """(rows, cols) CUDA view of x (rows x stride bits) starting `offset` elements into a buffer."""
    import torch

    rows, stride = x.shape
    sint = np.int32 if x.dtype == np.uint32 else np.int16
    flat = torch.zeros(offset + rows * stride + 8, dtype=torch.int32 if sint is np.int32 else torch.int16,
                       device="cuda")
    flat[offset: offset + rows * stride] = torch.from_numpy(np.ascontiguousarray(x).view(sint).ravel()).cuda()
    return flat.as_strided((rows, cols), (stride, 1), offset), flat


def gpu_select(x: np.ndarray, cols: int, k: int, dtype: str, plan: int = 0, offset: int = 0):
    import torch

    from wide_bf16_row_gb300 import topk

    view, hold = _device(x, cols, offset)
    idx, val, count, mask = topk.select_topk(view, k, dtype=CODES[dtype], plan=plan)
    torch.cuda.synchronize()
    bits = np.uint32 if dtype == "f32" else np.uint16
    out = (idx.cpu().numpy(), val.cpu().numpy().view(bits), count.cpu().numpy(), mask.cpu().numpy().view(np.uint32))
    del hold
    return out


def assert_same(got, exp, what):
    for g, e, name in zip(got, exp, ("idx", "val", "count", "mask")):
        if not np.array_equal(g, e):
            bad = np.argwhere(g != e)
            first = tuple(bad[0])
            raise AssertionError(f"{what}: {name} differs at {len(bad)} places, first {first}: "
                                 f"got {g[first]} expected {e[first]}")


def gen(dtype: str, rows: int, cols: int, seed: int, stride: int | None = None, **kw):
    if dtype == "bf16":
        return synth.mixed_rows(rows, cols, seed=seed, row_stride=stride, **kw)
    if dtype == "f16":
        return synth.mixed_rows_f16(rows, cols, seed=seed, row_stride=stride, **kw)
    return synth.mixed_rows_f32(rows, cols, seed=seed, row_stride=stride, **kw)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("k", [1, 20, 64, 65, 256, 1024])
def test_formats_and_k(dtype, k):
    """Mixed rows (specials, copies, subnormals) at several widths, padded strides."""
    for rows, cols, stride, seed in ((7, 5000, 5003, 1), (3, 70001, 70016, 2), (2, 700, 700, 3)):
        x = gen(dtype, rows, cols, seed + 10 * k, stride, special_frac=0.03, dup_frac=0.05)
        exp = oracle.topk(x, cols, k, dtype=dtype)
        assert_same(gpu_select(x, cols, k, dtype, plan=64), exp, f"{dtype} k{k} {rows}x{cols}")


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("offset", [1, 3, 5])
def test_unaligned_row_bases(dtype, offset):
    x = gen(dtype, 5, 3001, 40 + offset, 3011, special_frac=0.05)
    for k in (7, 300):
        assert_same(gpu_select(x, 3001, k, dtype, plan=64, offset=offset), oracle.topk(x, 3001, k, dtype=dtype),
                    f"{dtype} offset {offset} k{k}")


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_heavy_ties_take_the_exact_path(dtype):
    """More than 4096 columns reach the bound: all +-0 rows, three distinct
    values, a k-th key shared by thousands; plus all-NaN and short rows."""
    rng = np.random.default_rng(7)
    cols = 20000
    bits = np.uint32 if dtype == "f32" else np.uint16
    sign = (1 << 31) if dtype == "f32" else (1 << 15)
    one = {"bf16": 0x3F80, "f16": 0x3C00, "f32": 0x3F800000}[dtype]
    two = {"bf16": 0x4000, "f16": 0x4000, "f32": 0x40000000}[dtype]
    nan = {"bf16": 0x7FC0, "f16": 0x7E00, "f32": 0x7FC00000}[dtype]
    x = np.zeros((6, cols), bits)
    x[0] = rng.integers(0, 2, size=cols).astype(bits) * bits(sign)          # +-0 only
    x[1] = rng.choice(np.array([one, two, one | sign], bits), size=cols)      # three values
    x[2] = np.where(rng.random(cols) < 0.001, two, one).astype(bits)          # few 2.0, many 1.0
    x[3] = nan                                                                # all NaN
    x[4] = nan
    x[4, ::4000] = one                                                        # five numbers
    x[5] = rng.integers(0, 2, size=cols).astype(bits) * bits(sign)
    x[5, 100:110] = two
    for k in (1, 33, 64, 500, 1024):
        assert_same(gpu_select(x, cols, k, dtype, plan=64), oracle.topk(x, cols, k, dtype=dtype),
                    f"{dtype} ties k{k}")


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_rows_shorter_than_k(dtype):
    x = gen(dtype, 9, 37, 5, 40, special_frac=0.2)
    for k in (36, 37, 38, 1024):
        assert_same(gpu_select(x, 37, k, dtype, plan=64), oracle.topk(x, 37, k, dtype=dtype), f"{dtype} k{k}")


def test_bench_shape_through_the_wide_kernel():
    w = synth.config_draft_window()
    exp = oracle.topk(w.logits, w.cols, w.k)
    assert_same(gpu_select(w.logits, w.cols, w.k, "bf16", plan=64), exp, "256x248320 wide")
    for k in (100, 1024):
        exp = oracle.topk(w.logits[:16], w.cols, k)
        assert_same(gpu_select(w.logits[:16], w.cols, k, "bf16", plan=64), exp, f"16x248320 k{k}")


def test_specials_config_all_formats():
    """16 x 248320 with NaN, infinities, zeros, an all-NaN and an all-zero row (bf16),
    and fp16/fp32 rows of the same width."""
    w = synth.config_specials()
    assert_same(gpu_select(w.logits, w.cols, 300, "bf16", plan=64), oracle.topk(w.logits, w.cols, 300),
                "specials bf16 k300")
    for dtype in ("f16", "f32"):
        x = gen(dtype, 6, 248320, 77, 248384, special_frac=0.01, dup_frac=0.01)
        for k in (20, 1024):
            assert_same(gpu_select(x, 248320, k, dtype), oracle.topk(x, 248320, k, dtype=dtype),
                        f"{dtype} 248320 k{k}")


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_masked_rows_all_formats(dtype):
    """-inf masks (random, dense, a padded vocabulary's tail) with a few +inf,
    no NaN, through AUTO and the wide kernel: vectors whose only non-finite
    values are infinities skip the exact re-scan and keep their keys."""
    masks = ((0.1, 0, 0.0), (0.6, 0, 0.0), (0.0, 3000, 0.0), (0.1, 64, 0.0005))
    for i, (frac, tail, pinf) in enumerate(masks):
        cols = 70001 if i % 2 else 98592
        x = synth.masked_rows(24, cols, seed=31 + i, mask_frac=frac, tail=tail, plus_inf_frac=pinf,
                              row_stride=cols + 3 * (i % 2), fmt=dtype)
        for k in (20, 300, 1024):
            exp = oracle.topk(x, cols, k, dtype=dtype)
            for plan in (0, 64):
                assert_same(gpu_select(x, cols, k, dtype, plan=plan, offset=i % 3), exp,
                            f"{dtype} masked mask={frac} tail={tail} +inf={pinf} k{k} plan{plan}")


def _tie_groups(dtype: str, cols: int, groups, seed: int) -> np.ndarray:
    """Rows of small noise with exact copies of a few large values (count,
    value) at random columns, in the given format's bits."""
    rng = np.random.default_rng(seed)
    rows = []
    for r in range(4):
        v = rng.standard_normal(cols) * 0.5
        for count, value in groups:
            v[rng.choice(cols, size=count, replace=False)] = value
        rows.append(v)
    v = np.stack(rows)
    if dtype == "bf16":
        return synth.round_to_bf16(v.astype(np.float32))
    if dtype == "f16":
        return v.astype(np.float16).view(np.uint16)
    return v.astype(np.float32).view(np.uint32)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_wide_select_before_sort(dtype):
    """More than 1024 entries reach the wide kernel's bound: the k largest are
    selected before ranking -- ties at the k-th key ranked by column, k <= 512
    ranked directly, larger k sorted -- or, with more than 512 ties at the
    k-th key, all entries are sorted.  Each case against the oracle."""
    cases = [
        (((400, 5.0), (800, 4.0)), 300),               # the k-th key among 400 ties: ranked
        (((400, 5.0), (450, 4.0), (300, 3.5)), 500),   # 100 of 450 ties at 4.0
        (((700, 5.0), (400, 4.0)), 900),               # 200 of 400 ties: the 1024-entry sort
        (((300, 5.0), (900, 4.0)), 1000),              # 700 of 900 ties: more than 512, all sorted
        (((1100, 4.0),), 1024),                        # every entry a tie
    ]
    for i, (groups, k) in enumerate(cases):
        x = _tie_groups(dtype, 98592, groups, seed=100 + i)
        exp = oracle.topk(x, 98592, k, dtype=dtype)
        assert_same(gpu_select(x, 98592, k, dtype, plan=64), exp, f"{dtype} groups {groups} k{k}")


def test_bf16_small_k_matches_tf_topk_bf16():
    """tf_topk_select on bf16 with k <= 64 runs the tf_topk_bf16 plans: same bytes."""
    from tests.gpu_util import gpu_topk
    w = synth.config_draft_head()
    for plan in (0, 2, 8):
        got = gpu_select(w.logits, w.cols, w.k, "bf16", plan=plan)
        assert_same(got, gpu_topk(w.logits, w.cols, w.k, plan=plan), f"select plan {plan}")


@pytest.mark.parametrize("plan", [0, 1, 2, 4, 8, 16])
def test_f16_on_the_cluster_plans(plan):
    """fp16, k <= 64, on SINGLE and CLUSTER2..16 (and AUTO): mixed rows with every fp16
    special, padded strides, an unaligned row base, heavy ties (the exact
    path) and all-NaN rows, against the oracle."""
    x = gen("f16", 6, 70001, 3 + plan, 70016, special_frac=0.02, dup_frac=0.05)
    for k in (1, 20, 64):
        assert_same(gpu_select(x, 70001, k, "f16", plan=plan), oracle.topk(x, 70001, k, dtype="f16"),
                    f"f16 plan {plan} k{k}")
    assert_same(gpu_select(x, 70001, 33, "f16", plan=plan, offset=3), oracle.topk(x, 70001, 33, dtype="f16"),
                f"f16 plan {plan} offset 3")
    rng = np.random.default_rng(plan)
    ties = np.zeros((5, 40000), np.uint16)
    ties[0] = rng.integers(0, 2, size=40000).astype(np.uint16) << np.uint16(15)      # +-0
    ties[1] = rng.choice(np.array([0x3C00, 0x4000, 0xBC00], np.uint16), size=40000)  # three values
    ties[2] = 0x7E00                                                                 # all NaN
    ties[3] = rng.choice(np.array([0x7C00, 0xFC00, 0x0001, 0x8001], np.uint16), size=40000)  # infs, subnormals
    ties[4] = (rng.standard_normal(40000) * 2).astype(np.float16).view(np.uint16)
    for k in (1, 64):
        assert_same(gpu_select(ties, 40000, k, "f16", plan=plan), oracle.topk(ties, 40000, k, dtype="f16"),
                    f"f16 ties plan {plan} k{k}")


def test_f16_bench_shape_auto():
    """256 x 248320 fp16 (the bench workload's values rounded to fp16), AUTO plan."""
    w = synth.config_draft_window()
    with np.errstate(over="ignore"):
        x = synth.bf16_to_float(w.logits).astype(np.float16).view(np.uint16)
    assert_same(gpu_select(x, w.cols, w.k, "f16"), oracle.topk(x, w.cols, w.k, dtype="f16"), "f16 256x248320")


# fp32 with k <= 64 on AUTO runs the fp32 cluster kernel; the shapes pick its
# span counts 1 (few rows; a row per SM or more with rows of one chunk; many
# rows), 2, 4 and 8
F32_SHAPES = [(6, 5000, 5008), (3, 70001, 70016), (40, 40000, 40000), (160, 20000, 20004), (200, 8000, 8004),
              (1000, 3000, 3001)]


@pytest.mark.parametrize("rows,cols,stride", F32_SHAPES, ids=lambda v: str(v))
def test_f32_cluster_kernel(rows, cols, stride):
    """fp32, k <= 64, AUTO (the fp32 cluster kernel): mixed rows with every
    fp32 special, copies and low-half near-ties, padded strides, row bases
    off the 16-byte grid, against the oracle."""
    x = gen("f32", rows, cols, 11 + rows, stride, special_frac=0.02, dup_frac=0.05)
    for k in (1, 20, 33, 64):
        assert_same(gpu_select(x, cols, k, "f32"), oracle.topk(x, cols, k, dtype="f32"), f"f32 {rows}x{cols} k{k}")
    for offset in (1, 2, 3):
        assert_same(gpu_select(x, cols, 20, "f32", offset=offset), oracle.topk(x, cols, 20, dtype="f32"),
                    f"f32 {rows}x{cols} offset {offset}")


@pytest.mark.parametrize("cols", [5000, 70001])
def test_f32_cluster_kernel_ties_and_specials(cols):
    """Heavy ties (the exact path) and special rows on the fp32 cluster kernel."""
    rng = np.random.default_rng(cols)
    ties = np.zeros((6, cols), np.uint32)
    ties[0] = rng.integers(0, 2, size=cols).astype(np.uint32) << np.uint32(31)         # +-0
    ties[1] = rng.choice(np.array([0x3F800000, 0x40000000, 0xBF800000], np.uint32), size=cols)
    ties[2] = 0x7FC00000                                                               # all NaN
    ties[3] = rng.choice(np.array([0x7F800000, 0xFF800000, 0x00000001, 0x80000001, 0xFFFFFFFF], np.uint32),
                         size=cols)                                                    # infs, subnormals, a NaN
    ties[4] = (rng.standard_normal(cols) * 2).astype(np.float32).view(np.uint32)
    ties[5] = np.float32(-3.5).view(np.uint32)                                         # one negative value
    for k in (1, 20, 64):
        assert_same(gpu_select(ties, cols, k, "f32"), oracle.topk(ties, cols, k, dtype="f32"), f"f32 ties k{k}")


def test_f32_cluster_kernel_short_rows_and_bench_shape():
    """Rows shorter than k, and the bench workload's values widened to fp32
    (256 x 248320, AUTO) against the oracle and against the wide kernel."""
    x = gen("f32", 4, 37, 5, 40)
    assert_same(gpu_select(x, 37, 64, "f32"), oracle.topk(x, 37, 64, dtype="f32"), "f32 37 columns k64")
    w = synth.config_draft_window()
    x = (np.asarray(w.logits, np.uint32) << np.uint32(16)).astype(np.uint32)
    exp = oracle.topk(x[:32], w.cols, w.k, dtype="f32")
    got = gpu_select(x, w.cols, w.k, "f32")
    assert_same(tuple(a[:32] for a in got), exp, "f32 256x248320 (first 32 rows)")
    assert_same(got, gpu_select(x, w.cols, w.k, "f32", plan=64), "f32 256x248320 cluster vs wide")
