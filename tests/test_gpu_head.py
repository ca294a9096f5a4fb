"""GPU parity of the draft head with the top-k in its epilogue
(tf_topk_head_bf16) against the CPU oracle, byte for byte: the head's logits
are bf16(hidden . weight^T) with an fp32 sum (the reading of TensorFold PR
#713, change 3, whose top-k consumes the draft head's bf16 rows), and the
selection is the pages' top-k.  The seeded inputs make every sum exact in
fp32, so the result is unique.  Also: the same result from cuBLAS's product
followed by tf_topk_bf16, two calls on one workspace, and the guards."""
from __future__ import annotations

import numpy as np
import pytest

from oracle import head as head_oracle
from tests.gpu_util import assert_same
from wide_bf16_row_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from wide_bf16_row_gb300 import build
    build.build()


def _dev(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda")


def _np(res):
    import torch
    idx, val, count, mask = res
    torch.cuda.synchronize()
    return (idx.cpu().numpy(), val.view(torch.int16).cpu().numpy().view(np.uint16), count.cpu().numpy(),
            mask.cpu().numpy().view(np.uint32))


# rows, dim, vocab, k: the draft head; the wide shape as a head; a dim that is
# not a multiple of 64; a vocabulary that is not a multiple of 128; k above
# the vocabulary; one row; sixteen rows of eight dims
SHAPES = [
    (15, 2048, 98592, 16),
    (16, 2048, 248320, 64),
    (7, 136, 5000, 20),
    (16, 512, 257, 64),
    (2, 64, 1, 4),
    (1, 64, 100, 1),
    (16, 8, 129, 64),
    (5, 1024, 33000, 33),
    (3, 200, 70001, 8),
]


@pytest.mark.parametrize("rows,dim,vocab,k", SHAPES, ids=lambda v: str(v))
def test_head_matches_the_oracle(rows, dim, vocab, k):
    from wide_bf16_row_gb300 import topk

    h = synth.head_inputs(rows, dim, vocab, k, seed=rows * 1000 + dim + vocab + k)
    exp = head_oracle.topk(h.hidden, h.weight, k)
    got = _np(topk.head_topk_bf16(_dev(h.hidden), _dev(h.weight), k))
    assert_same(got, exp, f"head {rows}x{dim}x{vocab} k={k}")
    assert topk.device_fault() == 0


@pytest.mark.parametrize("vocab,k", [(98592, 16), (33000, 64), (200, 5)])
def test_head_all_logits_tied(vocab, k):
    """Every logit equal (one-hot hidden rows against a constant weight
    column): each row is the first k columns, across tiles and CTAs that
    select out of column order.  A row of zeros ties at +0."""
    from wide_bf16_row_gb300 import topk

    rows, dim = 4, 64
    one = synth.round_to_bf16(np.array([1.0], np.float32))[0]
    hidden = np.zeros((rows, dim), np.uint16)
    hidden[:3, 5] = one                                   # rows 0-2: logit = weight[:, 5]; row 3 all zero
    weight = np.zeros((vocab, dim), np.uint16)
    weight[:, 5] = synth.round_to_bf16(np.array([0.75], np.float32))[0]
    exp = head_oracle.topk(hidden, weight, k)
    assert exp[0][0].tolist() == list(range(min(k, vocab))) + [-1] * (k - min(k, vocab))
    got = _np(topk.head_topk_bf16(_dev(hidden), _dev(weight), k))
    assert_same(got, exp, f"tied head {vocab} k={k}")


def test_head_matches_cublas_then_topk():
    """cuBLAS's bf16 product (fp32 sum, rounded to bf16) followed by the
    ordinary top-k gives the same lists: the sums are exact."""
    import torch

    from wide_bf16_row_gb300 import topk

    h = synth.config_head_draft()
    hid, w = _dev(h.hidden).view(torch.bfloat16), _dev(h.weight).view(torch.bfloat16)
    logits = hid @ w.T
    two_step = _np(topk.topk_bf16(logits, h.k))
    fused = _np(topk.head_topk_bf16(hid, w, h.k))
    assert_same(fused, two_step, "fused head vs cuBLAS + tf_topk_bf16")


def test_two_calls_share_a_workspace():
    import torch

    from wide_bf16_row_gb300 import topk

    a = synth.head_inputs(15, 256, 40000, 16, seed=1)
    b = synth.head_inputs(9, 512, 7000, 64, seed=2)
    ws = torch.empty((topk.tf_topk_head_bf16_workspace(16, 64),), dtype=torch.uint8, device="cuda")
    ra = topk.head_topk_bf16(_dev(a.hidden), _dev(a.weight), a.k, workspace=ws)
    ea = head_oracle.topk(a.hidden, a.weight, a.k)
    assert_same(_np(ra), ea, "first call")
    rb = topk.head_topk_bf16(_dev(b.hidden), _dev(b.weight), b.k, workspace=ws)
    assert_same(_np(rb), head_oracle.topk(b.hidden, b.weight, b.k), "second call, same workspace")


def test_captured_call_replays():
    """A call captured in a CUDA graph, replayed on new inputs written into
    the same buffers (the cut-tile tickets are cleared by each call), matches
    the oracle every time."""
    import torch

    from wide_bf16_row_gb300 import topk

    rows, dim, vocab, k = 15, 512, 60000, 16
    first = synth.head_inputs(rows, dim, vocab, k, seed=21)
    hid, w = _dev(first.hidden), _dev(first.weight)
    ws = torch.empty((topk.tf_topk_head_bf16_workspace(rows, k),), dtype=torch.uint8, device="cuda")
    out = (torch.empty((rows, k), dtype=torch.int32, device="cuda"),
           torch.empty((rows, k), dtype=torch.int16, device="cuda"),
           torch.empty((rows,), dtype=torch.int32, device="cuda"),
           torch.empty((rows,), dtype=torch.int32, device="cuda"))
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        topk.head_topk_bf16(hid, w, k, out=out, workspace=ws, stream=side)  # warm: per-device setup
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        topk.head_topk_bf16(hid, w, k, out=out, workspace=ws, stream=side)
    for seed in (21, 22, 23, 23):
        h = synth.head_inputs(rows, dim, vocab, k, seed=seed)
        hid.copy_(_dev(h.hidden))
        w.copy_(_dev(h.weight))
        torch.cuda.synchronize()
        with torch.cuda.stream(side):
            graph.replay()
        torch.cuda.synchronize()
        assert_same(_np(out), head_oracle.topk(h.hidden, h.weight, k), f"replay, seed {seed}")
    assert topk.device_fault() == 0


def test_guards():
    import torch

    from wide_bf16_row_gb300 import topk

    h = _dev(np.zeros((4, 64), np.uint16))
    w = _dev(np.zeros((100, 64), np.uint16))
    out = [torch.full((4, 8), 5, dtype=torch.int32, device="cuda") for _ in range(2)] + \
          [torch.full((4,), 5, dtype=torch.int32, device="cuda") for _ in range(2)]
    small = torch.empty((8,), dtype=torch.uint8, device="cuda")

    def call(rows=4, dim=64, vocab=100, k=8, ws=None, nbytes=None, hp=None, wp=None):
        ws = ws if ws is not None else torch.empty((1 << 20,), dtype=torch.uint8, device="cuda")
        return topk.tf_topk_head_bf16(hp or h.data_ptr(), wp or w.data_ptr(), rows, dim, vocab, k, ws.data_ptr(),
                                      ws.numel() if nbytes is None else nbytes, out[0].data_ptr(),
                                      out[1].data_ptr(), out[2].data_ptr(), out[3].data_ptr(), None)

    assert call(k=65) == topk.ERR_K
    assert call(rows=17) == topk.ERR_SHAPE
    assert call(dim=12) == topk.ERR_SHAPE
    assert call(vocab=0) == topk.ERR_SHAPE
    assert call(hp=h.data_ptr() + 2) == topk.ERR_ALIGN
    assert call(ws=small) == topk.ERR_SCRATCH
    torch.cuda.synchronize()
    assert all(bool((t == 5).all()) for t in out)
    # the size the query gives is enough, and one byte less is refused, for a
    # vocabulary long enough to take every CTA of the grid (160 tiles of 128)
    need = topk.tf_topk_head_bf16_workspace(4, 8)
    assert need > 0
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    wide = _dev(np.zeros((160 * 128, 64), np.uint16))
    assert call(ws=ws, nbytes=need - 1, vocab=160 * 128, wp=wide.data_ptr()) == topk.ERR_SCRATCH
    assert call(ws=ws, nbytes=need, vocab=160 * 128, wp=wide.data_ptr()) == topk.OK
    torch.cuda.synchronize()
    assert topk.tf_topk_head_bf16_workspace(16, 64) >= need
