"""The allocation-free entry point, tf_topk_bf16_noalloc, against the CPU oracle.

Some callers cannot allocate device memory once they run: a serving engine
that has reserved nearly all of HBM for its caches, or a host of custom
operators that only passes in the buffers it owns.  For them the library keeps
its scratch in one static device array instead of allocating it per stream.
These checks call that entry point through the C ABI, two calls in a row on
one stream (the second reuses the array the first left behind), and require
byte-equal results with the CPU oracle -- the same bar as every other parity
test here.  One more check shows that the calls allocate nothing: the
device's free memory is the same before and after two calls on a new stream.

The file name sorts last, so a run that stops at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
from __future__ import annotations

import pytest

import oracle
from tests.gpu_util import assert_same, device_matrix, to_numpy
from wide_bf16_row_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from wide_bf16_row_gb300 import build
    build.build()


def _outputs(rows: int, k: int, fill: int = 0):
    import torch

    return (torch.full((rows, k), fill, dtype=torch.int32, device="cuda"),
            torch.full((rows, k), fill, dtype=torch.int16, device="cuda"),
            torch.full((rows,), fill, dtype=torch.int32, device="cuda"),
            torch.full((rows,), fill, dtype=torch.int32, device="cuda"))


def _call(fn, view, k: int, out, stream) -> int:
    rows, cols = view.shape
    return fn(view.data_ptr(), rows, cols, view.stride(0), k, out[0].data_ptr(), out[1].data_ptr(),
              out[2].data_ptr(), out[3].data_ptr(), stream.cuda_stream)


def _inputs():
    """Shapes that cut rows into pieces across CTAs (so the shared scratch is
    really used), one with fewer rows than CTAs, and a single short row."""
    yield synth.config_draft_window()            # 256 x 248320, k = 20
    yield synth.config_draft_head()              # 15 x 98592, k = 16
    yield synth.config_specials()                # 16 x 248320 (padded stride), k = 64
    yield synth.config_draft_single()            # 1 x 4096, k = 8


@pytest.mark.parametrize("w", list(_inputs()), ids=lambda w: w.name)
def test_two_calls_in_a_row_match_the_oracle(w):
    import torch

    from wide_bf16_row_gb300 import topk

    view, keep = device_matrix(w.logits, w.cols)
    s = torch.cuda.current_stream()
    exp = oracle.topk(w.logits, w.cols, w.k)
    first, second = _outputs(w.rows, w.k, fill=7), _outputs(w.rows, w.k, fill=9)
    assert _call(topk.tf_topk_bf16_noalloc, view, w.k, first, s) == topk.OK
    assert _call(topk.tf_topk_bf16_noalloc, view, w.k, second, s) == topk.OK
    assert_same(to_numpy(first), exp, f"{w.name} first no-alloc call")
    assert_same(to_numpy(second), exp, f"{w.name} second no-alloc call")
    assert topk.device_fault() == 0
    del keep


def test_calls_allocate_no_device_memory():
    """After one warm call (it loads the kernel and looks up the array's
    address), two more calls on a stream created for them leave the device's
    free memory unchanged."""
    import torch

    from wide_bf16_row_gb300 import topk

    w = synth.config_draft_window()
    view, keep = device_matrix(w.logits, w.cols)
    out = _outputs(w.rows, w.k)
    assert _call(topk.tf_topk_bf16_noalloc, view, w.k, out, torch.cuda.current_stream()) == topk.OK
    fresh = torch.cuda.Stream()
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for _ in range(2):
        assert _call(topk.tf_topk_bf16_noalloc, view, w.k, out, fresh) == topk.OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert_same(to_numpy(out), oracle.topk(w.logits, w.cols, w.k), "no-alloc call on a new stream")
    del keep


def test_back_to_back_calls_on_different_shapes():
    """Two different matrices, queued without a synchronisation in between."""
    import torch

    from wide_bf16_row_gb300 import topk

    a, b = synth.config_draft_window(), synth.config_draft_head()
    va, ka = device_matrix(a.logits, a.cols)
    vb, kb = device_matrix(b.logits, b.cols)
    s = torch.cuda.current_stream()
    na, nb = _outputs(a.rows, a.k, fill=3), _outputs(b.rows, b.k, fill=3)
    assert _call(topk.tf_topk_bf16_noalloc, va, a.k, na, s) == topk.OK
    assert _call(topk.tf_topk_bf16_noalloc, vb, b.k, nb, s) == topk.OK
    assert_same(to_numpy(na), oracle.topk(a.logits, a.cols, a.k), "256x248320 then ...")
    assert_same(to_numpy(nb), oracle.topk(b.logits, b.cols, b.k), "... 15x98592")
    del ka, kb


def test_guards_match_the_allocating_entry():
    import torch

    from wide_bf16_row_gb300 import topk

    x = torch.zeros((4, 100), dtype=torch.int16, device="cuda")
    out = _outputs(4, 8, fill=5)
    s = torch.cuda.current_stream()
    assert _call(topk.tf_topk_bf16_noalloc, x, 65, out, s) == topk.ERR_K
    assert topk.tf_topk_bf16_noalloc(x.data_ptr(), 4, 100, 99, 8, out[0].data_ptr(), out[1].data_ptr(),
                                     out[2].data_ptr(), out[3].data_ptr(), None) == topk.ERR_SHAPE
    assert topk.tf_topk_bf16_noalloc(x.data_ptr(), 0, 100, 100, 8, 0, 0, 0, 0, None) == topk.OK
    torch.cuda.synchronize()
    assert all(bool((t == 5).all()) for t in out)
    assert "TF_TOPK_NOALLOC_MAX_CTAS" in topk.strerror(topk.ERR_SCRATCH)
    # a 152-SM GB300 launches at most 304 CTAs: well inside the static area
    props = torch.cuda.get_device_properties(0)
    assert 2 * props.multi_processor_count <= 512
