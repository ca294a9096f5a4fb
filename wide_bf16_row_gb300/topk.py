"""Python binding over ``libtf_topk.so`` (C ABI in ``include/tf_topk.h``).

Argument marshalling only: every step runs in the library's CUDA kernels.
PyTorch supplies device memory and the current stream.  If the library has
not been built, every entry point raises -- there is no fallback.

Tensor-level calls: ``topk_bf16`` (bf16 rows, k <= 64, any launch plan),
``select_topk`` (bf16 / fp16 / fp32 rows, k <= 1024), ``merge_bf16``
(per-shard lists into each row's top k), ``nucleus_bf16`` (top-p
probabilities over the lists) and ``head_topk_bf16`` (the draft head's
product and the top-k in one kernel).  The raw C entry points are exposed under
their C names.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

PKG = Path(__file__).resolve().parent
LIBRARY = PKG / "libtf_topk.so"

# status codes (include/tf_topk.h)
OK, ERR_NULL, ERR_SHAPE, ERR_K, ERR_ALIGN, ERR_PLAN, ERR_DEVICE, ERR_CUDA = range(8)
ERR_SCRATCH = 8  # tf_topk_bf16_noalloc only
ERR_ARG = 9  # tf_topk_nucleus_bf16 only
ERR_DTYPE = 10  # tf_topk_select only
DTYPE_BF16, DTYPE_F16, DTYPE_F32 = 0, 1, 2
PLAN_WIDE = 64  # tf_topk_select_with_plan: the wide kernel

# launch plans (include/tf_topk.h)
PLAN_AUTO, PLAN_SINGLE, PLAN_STREAM = 0, 1, 32
PLAN_CLUSTER = {2: 2, 4: 4, 8: 8, 16: 16}
PLANS = (PLAN_AUTO, PLAN_SINGLE, 2, 4, 8, 16, PLAN_STREAM)

_lib = None


class TopkError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"tf_topk status {status}: {message}")
        self.status = status


def library() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it was never built."""
    global _lib
    if _lib is None:
        if not LIBRARY.exists():
            raise ImportError(f"{LIBRARY} is missing: build it with "
                              "`python -m wide_bf16_row_gb300.build` (no CPU fallback exists)")
        lib = ctypes.CDLL(str(LIBRARY))
        c_i64, c_i32, c_p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        lib.tf_topk_bf16.restype = ctypes.c_int
        lib.tf_topk_bf16.argtypes = [c_p, c_i64, c_i64, c_i64, c_i32, c_p, c_p, c_p, c_p, c_p]
        lib.tf_topk_bf16_with_plan.restype = ctypes.c_int
        lib.tf_topk_bf16_with_plan.argtypes = [c_p, c_i64, c_i64, c_i64, c_i32, c_p, c_p, c_p,
                                               c_p, c_i32, c_p]
        lib.tf_topk_merge_bf16.restype = ctypes.c_int
        lib.tf_topk_merge_bf16.argtypes = [c_p, c_p, c_p, c_p, c_i64, c_i32, c_i32, c_p, c_i32, c_p, c_p, c_p,
                                           c_p, c_p]
        lib.tf_topk_bf16_noalloc.restype = ctypes.c_int
        lib.tf_topk_bf16_noalloc.argtypes = [c_p, c_i64, c_i64, c_i64, c_i32, c_p, c_p, c_p, c_p, c_p]
        lib.tf_topk_nucleus_bf16.restype = ctypes.c_int
        lib.tf_topk_nucleus_bf16.argtypes = [c_p, c_p, c_i64, c_i32, ctypes.c_float, ctypes.c_float, c_p, c_p, c_p]
        lib.tf_topk_nucleus.restype = ctypes.c_int
        lib.tf_topk_nucleus.argtypes = [c_p, c_i32, c_p, c_i64, c_i32, ctypes.c_float, ctypes.c_float, c_p, c_p, c_p]
        lib.tf_topk_select.restype = ctypes.c_int
        lib.tf_topk_select.argtypes = [c_p, c_i32, c_i64, c_i64, c_i64, c_i32, c_p, c_p, c_p, c_p, c_p]
        lib.tf_topk_select_with_plan.restype = ctypes.c_int
        lib.tf_topk_select_with_plan.argtypes = [c_p, c_i32, c_i64, c_i64, c_i64, c_i32, c_p, c_p, c_p, c_p,
                                                 c_i32, c_p]
        lib.tf_topk_select_max_k.restype = c_i32
        lib.tf_topk_select_max_k.argtypes = []
        lib.tf_topk_device_fault.restype = ctypes.c_int
        lib.tf_topk_device_fault.argtypes = []
        lib.tf_topk_bf16_plan.restype = c_i32
        lib.tf_topk_bf16_plan.argtypes = [c_i64, c_i64, c_i32]
        for name in ("tf_topk_bf16_max_k", "tf_topk_bf16_max_spans", "tf_topk_bf16_cta_threads",
                     "tf_topk_bf16_chunk_columns"):
            getattr(lib, name).restype = c_i32
            getattr(lib, name).argtypes = []
        lib.tf_topk_head_bf16.restype = ctypes.c_int
        lib.tf_topk_head_bf16.argtypes = [c_p, c_p, c_i32, c_i32, c_i64, c_i32, c_p, ctypes.c_size_t, c_p, c_p,
                                          c_p, c_p, c_p]
        lib.tf_topk_head_bf16_workspace.restype = ctypes.c_size_t
        lib.tf_topk_head_bf16_workspace.argtypes = [c_i32, c_i32]
        lib.tf_topk_strerror.restype = ctypes.c_char_p
        lib.tf_topk_strerror.argtypes = [ctypes.c_int]
        lib.tf_topk_last_cuda_error.restype = ctypes.c_int
        lib.tf_topk_last_cuda_error.argtypes = []
        _lib = lib
    return _lib


def strerror(status: int) -> str:
    return library().tf_topk_strerror(status).decode()


def constants() -> dict:
    lib = library()
    return {
        "max_k": lib.tf_topk_bf16_max_k(),
        "max_spans": lib.tf_topk_bf16_max_spans(),
        "cta_threads": lib.tf_topk_bf16_cta_threads(),
        "chunk_columns": lib.tf_topk_bf16_chunk_columns(),
    }


MAX_K = 64


_raw_stream = None


def _stream_handle(stream, dev) -> int:
    """The cudaStream_t of ``stream``, or of the current stream of ``dev``
    (read through torch's raw-stream query where it has one: a plain
    ``torch.cuda.current_stream`` costs microseconds a call)."""
    global _raw_stream
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is None:
        import torch
        f = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        _raw_stream = f if f is not None else (lambda i: torch.cuda.current_stream(i).cuda_stream)
    return _raw_stream(dev.index)


def _on_device(dev, fn, *args):
    """fn(*args) with ``dev`` the current CUDA device (the library launches on
    the current device); the device is switched only when it is not already."""
    import torch
    if torch.cuda.current_device() == dev.index:
        return fn(*args)
    with torch.cuda.device(dev):
        return fn(*args)


def _check(status: int) -> None:
    if status != OK:
        msg = strerror(status)
        if status == ERR_CUDA:
            msg += f" (cudaError {library().tf_topk_last_cuda_error()})"
        raise TopkError(status, msg)


def tf_topk_bf16(logits: int, rows: int, cols: int, row_stride: int, k: int, out_idx: int,
                 out_val: int, out_count: int, out_nonfinite_mask: int, stream: int | None) -> int:
    """The C entry point with raw pointers (ints); returns the status code."""
    return library().tf_topk_bf16(logits, rows, cols, row_stride, k, out_idx, out_val, out_count,
                                  out_nonfinite_mask, stream)


def tf_topk_bf16_with_plan(logits: int, rows: int, cols: int, row_stride: int, k: int,
                           out_idx: int, out_val: int, out_count: int, out_nonfinite_mask: int,
                           plan: int, stream: int | None) -> int:
    """The C entry point with an explicit launch plan; returns the status code."""
    return library().tf_topk_bf16_with_plan(logits, rows, cols, row_stride, k, out_idx, out_val,
                                            out_count, out_nonfinite_mask, plan, stream)


def tf_topk_bf16_noalloc(logits: int, rows: int, cols: int, row_stride: int, k: int,
                         out_idx: int, out_val: int, out_count: int, out_nonfinite_mask: int,
                         stream: int | None) -> int:
    """The allocation-free C entry point (static scratch shared by every call;
    calls that overlap on the GPU race); returns the status code."""
    return library().tf_topk_bf16_noalloc(logits, rows, cols, row_stride, k, out_idx, out_val,
                                          out_count, out_nonfinite_mask, stream)


def tf_topk_merge_bf16(in_idx: int, in_val: int, in_count: int, in_mask: int, rows: int, shards: int,
                       k_in: int, shard_offset, k: int, out_idx: int, out_val: int, out_count: int,
                       out_mask: int, stream: int | None) -> int:
    """The C merge entry point; `shard_offset` is a host sequence of ints (or
    None to pass NULL).  Returns the status code."""
    off = None
    if shard_offset is not None:
        off = (ctypes.c_int64 * max(1, len(shard_offset)))(*[int(v) for v in shard_offset])
    return library().tf_topk_merge_bf16(in_idx, in_val, in_count, in_mask, rows, shards, k_in, off, k,
                                        out_idx, out_val, out_count, out_mask, stream)


def merge_bf16(idx, val, count, mask, offsets, k: int, *, out=None, stream=None):
    """Merge per-shard top lists into each row's top k.

    idx int32 [shards, rows, k_in], val bf16/int16/uint16 [shards, rows, k_in],
    count int32 [shards, rows], mask int32/uint32 [shards, rows] (all CUDA,
    contiguous), offsets: the column offset of each shard (host ints).
    Returns (idx int32 [rows, k], val [rows, k], count int32 [rows], mask int32 [rows]).
    """
    import torch

    shards, rows, k_in = idx.shape
    for t in (idx, val, count, mask):
        if not t.is_cuda or not t.is_contiguous():
            raise TopkError(ERR_SHAPE, "merge inputs must be contiguous CUDA tensors")
    if out is None:
        dev = idx.device
        out = (torch.empty((rows, k), dtype=torch.int32, device=dev),
               torch.empty((rows, k), dtype=val.dtype, device=dev),
               torch.empty((rows,), dtype=torch.int32, device=dev),
               torch.empty((rows,), dtype=torch.int32, device=dev))
    _check(_on_device(idx.device, tf_topk_merge_bf16, idx.data_ptr(), val.data_ptr(), count.data_ptr(),
                      mask.data_ptr(), rows, shards, k_in, list(offsets), k, out[0].data_ptr(), out[1].data_ptr(),
                      out[2].data_ptr(), out[3].data_ptr(), _stream_handle(stream, idx.device)))
    return out


def tf_topk_nucleus_bf16(val: int, count: int, rows: int, k: int, temperature: float, top_p: float,
                         out_prob: int, out_keep: int, stream: int | None) -> int:
    """The C nucleus (top-p) entry point with raw pointers; returns the status code."""
    return library().tf_topk_nucleus_bf16(val, count, rows, k, temperature, top_p, out_prob, out_keep, stream)


def tf_topk_nucleus(val: int, dtype: int, count: int, rows: int, k: int, temperature: float, top_p: float,
                    out_prob: int, out_keep: int, stream: int | None) -> int:
    """The C nucleus (top-p) entry point for lists of any format; returns the status code."""
    return library().tf_topk_nucleus(val, dtype, count, rows, k, temperature, top_p, out_prob, out_keep, stream)


def nucleus_bf16(val, count, temperature: float, top_p: float, *, out=None, stream=None):
    """Sampling probabilities over top-k lists (softmax of value / T, then the
    shortest best-first prefix with mass >= top_p, renormalised).

    val bf16/int16/uint16 [rows, k] and count int32 [rows] as ``topk_bf16``
    returns them (contiguous CUDA tensors).  Returns (prob float32 [rows, k],
    keep int32 [rows]).
    """
    return nucleus(val, count, temperature, top_p, dtype=DTYPE_BF16, out=out, stream=stream)


def nucleus(val, count, temperature: float, top_p: float, *, dtype: int | None = None, out=None, stream=None):
    """``nucleus_bf16`` for lists of any format ``select_topk`` returns:
    val bfloat16 / float16 / float32 [rows, k] (or int16 / int32 bits with
    ``dtype``), count int32 [rows]."""
    import torch

    codes = {torch.bfloat16: DTYPE_BF16, torch.float16: DTYPE_F16, torch.float32: DTYPE_F32,
             torch.int16: DTYPE_BF16, torch.uint16: DTYPE_BF16, torch.int32: DTYPE_F32}
    if dtype is None:
        if val.dtype not in codes:
            raise TypeError(f"unsupported list dtype {val.dtype}")
        dtype = codes[val.dtype]
    if val.element_size() != (4 if dtype == DTYPE_F32 else 2):
        raise TypeError("element size does not match dtype")
    if val.dim() != 2 or count.dim() != 1 or count.shape[0] != val.shape[0]:
        raise ValueError("val must be [rows, k] and count [rows]")
    for t in (val, count):
        if not t.is_cuda or not t.is_contiguous():
            raise TopkError(ERR_SHAPE, "nucleus inputs must be contiguous CUDA tensors")
    rows, k = val.shape
    if out is None:
        out = (torch.empty((rows, k), dtype=torch.float32, device=val.device),
               torch.empty((rows,), dtype=torch.int32, device=val.device))
    _check(_on_device(val.device, tf_topk_nucleus, val.data_ptr(), dtype, count.data_ptr(), rows, k,
                      float(temperature), float(top_p), out[0].data_ptr(), out[1].data_ptr(),
                      _stream_handle(stream, val.device)))
    return out


def tf_topk_select(logits: int, dtype: int, rows: int, cols: int, row_stride: int, k: int, out_idx: int,
                   out_val: int, out_count: int, out_nonfinite_mask: int, stream: int | None) -> int:
    """The C entry point for bf16 / fp16 / fp32 rows and k up to 1024; returns the status code."""
    return library().tf_topk_select(logits, dtype, rows, cols, row_stride, k, out_idx, out_val, out_count,
                                    out_nonfinite_mask, stream)


def tf_topk_select_with_plan(logits: int, dtype: int, rows: int, cols: int, row_stride: int, k: int,
                             out_idx: int, out_val: int, out_count: int, out_nonfinite_mask: int, plan: int,
                             stream: int | None) -> int:
    """tf_topk_select with a plan (0 AUTO, PLAN_WIDE, or a bf16 plan for k <= 64)."""
    return library().tf_topk_select_with_plan(logits, dtype, rows, cols, row_stride, k, out_idx, out_val,
                                              out_count, out_nonfinite_mask, plan, stream)


def select_topk(x, k: int, *, dtype: int | None = None, plan: int = 0, out=None, stream=None):
    """Exact top-k of every row of a CUDA bf16 / fp16 / fp32 matrix, k up to 1024.

    ``x``: bfloat16, float16 or float32 (or int16 / int32 holding the bits,
    with ``dtype`` one of DTYPE_*), 1-D or 2-D with unit column stride.
    Returns ``(idx int32[rows,k], val[rows,k] (x's dtype), count int32[rows],
    mask int32[rows])``.
    """
    import torch

    codes = {torch.bfloat16: DTYPE_BF16, torch.float16: DTYPE_F16, torch.float32: DTYPE_F32}
    if not x.is_cuda:
        raise ValueError("select_topk needs a CUDA tensor (no CPU path exists)")
    if dtype is None:
        if x.dtype not in codes:
            raise TypeError(f"pass dtype= for a {x.dtype} tensor of bits")
        dtype = codes[x.dtype]
    if x.element_size() != (4 if dtype == DTYPE_F32 else 2):
        raise TypeError("element size does not match dtype")
    if x.dim() == 1:
        x = x.unsqueeze(0)
    if x.dim() != 2 or (x.shape[1] > 1 and x.stride(1) != 1):
        raise ValueError("x must be 1-D or 2-D with contiguous columns")
    rows, cols = x.shape
    row_stride = x.stride(0) if rows > 1 else max(cols, x.stride(0))
    dev = x.device
    if out is None:
        out = (torch.empty((rows, k), dtype=torch.int32, device=dev),
               torch.empty((rows, k), dtype=x.dtype, device=dev),
               torch.empty((rows,), dtype=torch.int32, device=dev),
               torch.empty((rows,), dtype=torch.int32, device=dev))
    _check(_on_device(dev, tf_topk_select_with_plan, x.data_ptr(), dtype, rows, cols, row_stride, k,
                      out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(), out[3].data_ptr(), plan,
                      _stream_handle(stream, dev)))
    return out


HEAD_MAX_ROWS = 16


def tf_topk_head_bf16(hidden: int, weight: int, rows: int, dim: int, vocab: int, k: int, workspace: int,
                      workspace_bytes: int, out_idx: int, out_val: int, out_count: int, out_mask: int,
                      stream: int | None) -> int:
    """The fused draft-head entry point with raw pointers; returns the status code."""
    return library().tf_topk_head_bf16(hidden, weight, rows, dim, vocab, k, workspace, workspace_bytes, out_idx,
                                       out_val, out_count, out_mask, stream)


def tf_topk_head_bf16_workspace(rows: int, k: int) -> int:
    """Workspace bytes tf_topk_head_bf16 needs on the current device (0 for bad arguments)."""
    return library().tf_topk_head_bf16_workspace(rows, k)


def head_topk_bf16(hidden, weight, k: int, *, out=None, workspace=None, stream=None):
    """Top-k of every row of the draft head's logits, bf16(hidden @ weight.T),
    computed and selected in one kernel (the logits are never stored).

    ``hidden``: CUDA bf16 (or int16 bits) [rows, dim], rows <= 16;
    ``weight``: CUDA bf16 (or int16 bits) [vocab, dim]; both contiguous.
    Returns ``(idx int32[rows,k], val bfloat16[rows,k], count int32[rows],
    mask int32[rows])`` as ``topk_bf16`` gives them for the logit matrix.
    ``workspace``: a CUDA uint8 tensor of at least
    ``tf_topk_head_bf16_workspace(rows, k)`` bytes (allocated here if None).
    """
    import torch

    for t in (hidden, weight):
        if not t.is_cuda or not t.is_contiguous() or t.dim() != 2:
            raise ValueError("hidden and weight must be contiguous 2-D CUDA tensors")
        if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
            raise TypeError(f"expected bf16 bits, got {t.dtype}")
    rows, dim = hidden.shape
    vocab = weight.shape[0]
    if weight.shape[1] != dim:
        raise ValueError("hidden and weight disagree on dim")
    dev = hidden.device
    if out is None:
        out = (torch.empty((rows, k), dtype=torch.int32, device=dev),
               torch.empty((rows, k), dtype=torch.bfloat16, device=dev),
               torch.empty((rows,), dtype=torch.int32, device=dev),
               torch.empty((rows,), dtype=torch.int32, device=dev))
    if workspace is None:
        need = _on_device(dev, tf_topk_head_bf16_workspace, rows, k) if 1 <= rows <= HEAD_MAX_ROWS else 0
        workspace = torch.empty((max(need, 8),), dtype=torch.uint8, device=dev)
    _check(_on_device(dev, tf_topk_head_bf16, hidden.data_ptr(), weight.data_ptr(), rows, dim, vocab, k,
                      workspace.data_ptr(), workspace.numel(), out[0].data_ptr(), out[1].data_ptr(),
                      out[2].data_ptr(), out[3].data_ptr(), _stream_handle(stream, dev)))
    return out


def device_fault() -> int:
    """0, or the fault code a kernel recorded since the last check (then cleared)."""
    r = library().tf_topk_device_fault()
    if r < 0:
        _check(-r)
    return r


def plan(rows: int, cols: int, k: int) -> int:
    """Launch plan (TF_TOPK_PLAN_* code) the library picks for a shape on the current device."""
    r = library().tf_topk_bf16_plan(rows, cols, k)
    if r < 0:
        _check(-r)
    return r


def topk_bf16(x, k: int, *, plan: int = 0, out=None, stream=None):
    """Exact top-k of every row of a CUDA bf16 matrix.

    ``x``: a CUDA tensor of dtype bfloat16 (or int16/uint16 holding bf16 bits),
    1-D (one row) or 2-D with unit column stride; ``x.stride(0)`` is the row
    stride, so a column-sliced view of a padded buffer works as is.
    Returns ``(idx int32[rows,k], val bfloat16[rows,k], count int32[rows],
    mask int32[rows])``; ``mask`` holds the uint32 bits (1 NaN, 2 +inf, 4 -inf).
    ``out`` may supply those four tensors.  Runs on ``stream`` (a
    ``torch.cuda.Stream``) or the current stream of ``x``'s device.  ``plan``
    picks the launch plan (``PLANS``; 0 = the library's choice); every plan
    gives the same result.
    """
    import torch

    if not x.is_cuda:
        raise ValueError("topk_bf16 needs a CUDA tensor (no CPU path exists)")
    if x.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"expected bf16 bits, got {x.dtype}")
    if x.dim() == 1:
        x = x.unsqueeze(0)
    if x.dim() != 2:
        raise ValueError("x must be 1-D or 2-D")
    rows, cols = x.shape
    if cols > 1 and x.stride(1) != 1:
        raise ValueError("columns must be contiguous (stride(1) == 1)")
    row_stride = x.stride(0) if rows > 1 else max(cols, x.stride(0))
    dev = x.device
    if out is None:
        idx = torch.empty((rows, k), dtype=torch.int32, device=dev)
        val = torch.empty((rows, k), dtype=torch.bfloat16, device=dev)
        count = torch.empty((rows,), dtype=torch.int32, device=dev)
        mask = torch.empty((rows,), dtype=torch.int32, device=dev)
    else:
        idx, val, count, mask = out
        for t, shape, dtypes in ((idx, (rows, k), (torch.int32,)),
                                 (val, (rows, k), (torch.bfloat16, torch.int16, torch.uint16)),
                                 (count, (rows,), (torch.int32,)),
                                 (mask, (rows,), (torch.int32, torch.uint32))):
            if tuple(t.shape) != shape or t.dtype not in dtypes or not t.is_contiguous() \
                    or t.device != dev:
                raise ValueError("out tensors must be contiguous, on x's device, with shapes "
                                 "(rows,k), (rows,k), (rows,), (rows,)")
    _check(_on_device(dev, library().tf_topk_bf16_with_plan, x.data_ptr(), rows, cols, row_stride, k,
                      idx.data_ptr(), val.data_ptr(), count.data_ptr(), mask.data_ptr(), plan,
                      _stream_handle(stream, dev)))
    return idx, val, count, mask
