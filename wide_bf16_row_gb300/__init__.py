"""Exact per-row top-k over wide bf16 logit rows, on GB300 (sm_103a).

The compute path is the CUDA library ``libtf_topk.so`` (C ABI declared in
``include/tf_topk.h``); ``wide_bf16_row_gb300.topk`` is the thin Python binding
over it.  Importing the package itself loads nothing: ``synth`` (seeded input
generators) stays usable without a GPU, and the binding is loaded on first use
of one of its names.
"""
from __future__ import annotations

__all__ = ["topk_bf16", "tf_topk_bf16", "tf_topk_bf16_with_plan", "MAX_K", "TopkError", "PLANS"]


def __getattr__(name):
    if name in __all__:
        from . import topk as _topk
        return getattr(_topk, name)
    raise AttributeError(name)
