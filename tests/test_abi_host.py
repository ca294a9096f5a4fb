"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/tf_topk.h declares, its compile-time constants match
the header (the kernel/host constant tie of TensorFold PR #713, change 3), and
the argument guards ("Row ABI and guards" in the PR's "Exactness" table)
reject bad calls before any CUDA work."""
from __future__ import annotations

import ctypes
import re
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "tf_topk.h"


@pytest.fixture(scope="module")
def lib():
    from wide_bf16_row_gb300 import build
    build.build()
    from wide_bf16_row_gb300 import topk
    return topk.library()


def declared_functions() -> list[str]:
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tf_topk_\w+)\s*\(", text)))


def header_macros() -> dict[str, int]:
    out = {}
    for name, val in re.findall(r"#define\s+(TF_TOPK_\w+)\s+(\d+)", HEADER.read_text()):
        out[name] = int(val)
    return out


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "tf_topk_bf16" in names and len(names) >= 8
    for name in names:
        assert hasattr(lib, name), f"{name} declared in tf_topk.h but not exported"
    nm = subprocess.run(["nm", "-D", "--defined-only", str(ROOT / "wide_bf16_row_gb300" / "libtf_topk.so")],
                        capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (tf_topk_\w+)", nm))
    assert set(names) <= exported


def test_constants_match_header(lib):
    from wide_bf16_row_gb300 import topk
    macros = header_macros()
    c = topk.constants()
    assert c["max_k"] == macros["TF_TOPK_MAX_K"] == topk.MAX_K
    assert c["max_spans"] == macros["TF_TOPK_MAX_SPANS"]
    assert c["cta_threads"] % 32 == 0
    assert c["chunk_columns"] <= 65536 and c["chunk_columns"] % (8 * c["cta_threads"]) == 0
    for name, val in (("TF_TOPK_PLAN_AUTO", 0), ("TF_TOPK_PLAN_SINGLE", 1), ("TF_TOPK_PLAN_CLUSTER2", 2),
                      ("TF_TOPK_PLAN_CLUSTER4", 4), ("TF_TOPK_PLAN_CLUSTER8", 8),
                      ("TF_TOPK_PLAN_CLUSTER16", 16), ("TF_TOPK_PLAN_STREAM", 32)):
        assert macros[name] == val and val in topk.PLANS
    for i, name in enumerate(["TF_TOPK_OK", "TF_TOPK_ERR_NULL", "TF_TOPK_ERR_SHAPE", "TF_TOPK_ERR_K",
                              "TF_TOPK_ERR_ALIGN", "TF_TOPK_ERR_PLAN", "TF_TOPK_ERR_DEVICE",
                              "TF_TOPK_ERR_CUDA"]):
        assert macros[name] == i
        assert getattr(topk, name.replace("TF_TOPK_", "")) == i


FAKE = 0x10000  # a non-NULL, aligned address; guards reject before it is touched


def call(lib, logits=FAKE, rows=4, cols=100, stride=100, k=8, idx=FAKE, val=FAKE, count=FAKE,
         mask=FAKE, plan=None):
    if plan is None:
        return lib.tf_topk_bf16(logits, rows, cols, stride, k, idx, val, count, mask, None)
    return lib.tf_topk_bf16_with_plan(logits, rows, cols, stride, k, idx, val, count, mask, plan, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(k=0), 3), (dict(k=65), 3), (dict(k=-1), 3),
    (dict(cols=0), 2), (dict(rows=-1), 2), (dict(stride=99), 2), (dict(cols=2**31, stride=2**31), 2),
    (dict(rows=2**40, stride=2**30, cols=100), 2),
    (dict(logits=None), 1), (dict(idx=None), 1), (dict(val=None), 1), (dict(count=None), 1),
    (dict(mask=None), 1),
    (dict(logits=FAKE + 1), 4), (dict(idx=FAKE + 2), 4), (dict(val=FAKE + 1), 4),
    (dict(count=FAKE + 2), 4), (dict(mask=FAKE + 1), 4),
    (dict(plan=3), 5), (dict(plan=64), 5), (dict(plan=-1), 5), (dict(plan=17), 5),
])
def test_guards_reject_before_launch(lib, kwargs, status):
    assert call(lib, **kwargs) == status


def test_zero_rows_is_a_no_op(lib):
    assert call(lib, rows=0, logits=None, idx=None, val=None, count=None, mask=None) == 0
    assert call(lib, rows=0, plan=16) == 0
    assert call(lib, rows=0, plan=32) == 0


def test_strerror_covers_every_status(lib):
    from wide_bf16_row_gb300 import topk
    texts = {topk.strerror(s) for s in range(11)}
    assert len(texts) == 11 and "unknown status" not in texts
    assert topk.strerror(99) == "unknown status"


def test_product_path_never_touches_the_oracle():
    """The CUDA library and the binding share no code with the oracle."""
    pkg = ROOT / "wide_bf16_row_gb300"
    for p in list(pkg.rglob("*.py")) + list(pkg.rglob("*.cu")) + list(pkg.rglob("*.h")):
        text = p.read_text()
        assert "import oracle" not in text and "from oracle" not in text, p
        assert "topk_oracle" not in text, p
    nm = subprocess.run(["nm", "-D", str(pkg / "libtf_topk.so")], capture_output=True, text=True).stdout
    assert "oracle" not in nm


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    from wide_bf16_row_gb300 import topk
    monkeypatch.setattr(topk, "_lib", None)
    monkeypatch.setattr(topk, "LIBRARY", tmp_path / "missing.so")
    with pytest.raises(ImportError):
        topk.library()


def merge_call(lib, rows=4, shards=2, k_in=8, offsets=(0, 100), k=8, in_idx=FAKE, in_val=FAKE, count=FAKE,
               mask=FAKE, out_idx=FAKE, out_val=FAKE, out_count=FAKE, out_mask=FAKE):
    from wide_bf16_row_gb300 import topk
    return topk.tf_topk_merge_bf16(in_idx, in_val, count, mask, rows, shards, k_in, offsets, k, out_idx,
                                   out_val, out_count, out_mask, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(k=0), 3), (dict(k=65), 3), (dict(k_in=0), 3), (dict(k_in=65), 3),
    (dict(shards=0, offsets=(0,)), 2), (dict(shards=65, offsets=tuple(range(65))), 2), (dict(rows=-1), 2),
    (dict(offsets=(0, -1)), 2), (dict(offsets=(0, 2**31)), 2),
    (dict(in_idx=None), 1), (dict(in_val=None), 1), (dict(count=None), 1), (dict(mask=None), 1),
    (dict(out_idx=None), 1), (dict(out_val=None), 1), (dict(out_count=None), 1), (dict(out_mask=None), 1),
    (dict(offsets=None), 1),
    (dict(in_idx=FAKE + 2), 4), (dict(in_val=FAKE + 1), 4), (dict(count=FAKE + 2), 4), (dict(mask=FAKE + 1), 4),
    (dict(out_idx=FAKE + 2), 4), (dict(out_val=FAKE + 1), 4),
])
def test_merge_guards_reject_before_launch(lib, kwargs, status):
    """tf_topk_merge_bf16 checks its arguments before any CUDA work."""
    assert merge_call(lib, **kwargs) == status


def test_merge_zero_rows_is_a_no_op(lib):
    assert merge_call(lib, rows=0, in_idx=None, in_val=None, count=None, mask=None, out_idx=None,
                      out_val=None, out_count=None, out_mask=None) == 0


def nucleus_call(lib, rows=4, k=8, temperature=0.7, top_p=0.95, val=FAKE, count=FAKE, prob=FAKE, keep=FAKE):
    from wide_bf16_row_gb300 import topk
    return topk.tf_topk_nucleus_bf16(val, count, rows, k, temperature, top_p, prob, keep, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(temperature=-0.5), 9), (dict(temperature=float("nan")), 9), (dict(temperature=float("inf")), 9),
    (dict(top_p=0.0), 9), (dict(top_p=-1.0), 9), (dict(top_p=1.5), 9), (dict(top_p=float("nan")), 9),
    (dict(k=0), 3), (dict(k=65), 3), (dict(rows=-1), 2),
    (dict(val=None), 1), (dict(count=None), 1), (dict(prob=None), 1), (dict(keep=None), 1),
    (dict(val=FAKE + 1), 4), (dict(count=FAKE + 2), 4), (dict(prob=FAKE + 2), 4), (dict(keep=FAKE + 1), 4),
])
def test_nucleus_guards_reject_before_launch(lib, kwargs, status):
    """tf_topk_nucleus_bf16 checks its arguments before any CUDA work."""
    assert nucleus_call(lib, **kwargs) == status


def test_nucleus_zero_rows_is_a_no_op(lib):
    assert nucleus_call(lib, rows=0, val=None, count=None, prob=None, keep=None) == 0
    assert nucleus_call(lib, rows=0, temperature=0.0, top_p=1.0) == 0


def select_call(lib, dtype=0, rows=4, cols=100, stride=100, k=8, logits=FAKE, idx=FAKE, val=FAKE, count=FAKE,
                mask=FAKE, plan=0):
    from wide_bf16_row_gb300 import topk
    return topk.tf_topk_select_with_plan(logits, dtype, rows, cols, stride, k, idx, val, count, mask, plan, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(dtype=3), 10), (dict(dtype=-1), 10),
    (dict(k=0), 3), (dict(k=1025), 3), (dict(dtype=2, k=1025), 3),
    (dict(rows=-1), 2), (dict(cols=0), 2), (dict(stride=99), 2),
    (dict(dtype=1, plan=32), 5), (dict(dtype=1, k=65, plan=2), 5), (dict(dtype=1, k=65, plan=1), 5),
    (dict(k=65, plan=2), 5), (dict(plan=3), 5), (dict(dtype=2, plan=32), 5), (dict(dtype=2, plan=2), 5),
    (dict(logits=None), 1), (dict(idx=None), 1), (dict(val=None), 1), (dict(count=None), 1), (dict(mask=None), 1),
    (dict(logits=FAKE + 1), 4), (dict(dtype=2, logits=FAKE + 2), 4), (dict(dtype=2, val=FAKE + 2), 4),
    (dict(dtype=1, val=FAKE + 1), 4), (dict(idx=FAKE + 2), 4),
])
def test_select_guards_reject_before_launch(lib, kwargs, status):
    """tf_topk_select checks its arguments before any CUDA work."""
    assert select_call(lib, **kwargs) == status


def test_select_zero_rows_and_constants(lib):
    from wide_bf16_row_gb300 import topk
    assert select_call(lib, rows=0, logits=None, idx=None, val=None, count=None, mask=None) == 0
    assert select_call(lib, rows=0, dtype=2, k=1024, plan=64) == 0
    macros = header_macros()
    assert topk.library().tf_topk_select_max_k() == macros["TF_TOPK_MAX_K_WIDE"] == 1024
    assert (macros["TF_TOPK_DTYPE_BF16"], macros["TF_TOPK_DTYPE_F16"], macros["TF_TOPK_DTYPE_F32"]) == \
        (topk.DTYPE_BF16, topk.DTYPE_F16, topk.DTYPE_F32)
    assert macros["TF_TOPK_PLAN_WIDE"] == topk.PLAN_WIDE and macros["TF_TOPK_ERR_DTYPE"] == topk.ERR_DTYPE


def test_nucleus_any_format_guards(lib):
    from wide_bf16_row_gb300 import topk
    call = lambda **kw: topk.tf_topk_nucleus(kw.get("val", FAKE), kw.get("dtype", 2), FAKE, kw.get("rows", 4),
                                             kw.get("k", 8), 0.7, 0.95, FAKE, FAKE, None)
    assert call(dtype=3) == topk.ERR_DTYPE and call(dtype=-1) == topk.ERR_DTYPE
    assert call(val=FAKE + 2) == topk.ERR_ALIGN and call(dtype=1, val=FAKE + 1) == topk.ERR_ALIGN
    assert call(k=65) == topk.ERR_K and call(rows=0) == topk.OK


@pytest.mark.parametrize("kwargs,status", [
    ({"k": 0}, 3), ({"k": 65}, 3), ({"rows": 0}, 2), ({"rows": 17}, 2), ({"dim": 4}, 2), ({"dim": 12}, 2),
    ({"vocab": 0}, 2), ({"hidden": 0}, 1), ({"workspace": 0}, 1), ({"weight": FAKE + 8}, 4),
    ({"workspace": FAKE + 4}, 4), ({"val": FAKE + 1}, 4),
])
def test_head_guards_reject_before_any_cuda_work(lib, kwargs, status):
    """tf_topk_head_bf16's argument checks run before the device is touched."""
    a = {"hidden": FAKE, "weight": FAKE, "rows": 15, "dim": 2048, "vocab": 98592, "k": 16, "workspace": FAKE,
         "idx": FAKE, "val": FAKE, "count": FAKE, "mask": FAKE}
    a.update(kwargs)
    assert lib.tf_topk_head_bf16(a["hidden"], a["weight"], a["rows"], a["dim"], a["vocab"], a["k"], a["workspace"],
                                 1 << 30, a["idx"], a["val"], a["count"], a["mask"], None) == status


def test_head_workspace_query_rejects_bad_arguments(lib):
    assert lib.tf_topk_head_bf16_workspace(0, 16) == 0
    assert lib.tf_topk_head_bf16_workspace(17, 16) == 0
    assert lib.tf_topk_head_bf16_workspace(4, 65) == 0
