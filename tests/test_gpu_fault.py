"""A bounded wait that runs out, on the GPU, without a fault.

A test build of the library (macro TF_TOPK_TEST_WAIT_TIMEOUT, a separate
``libtf_topk_wait_timeout.so``) makes every stream-plan CTA wait, after its
first chunk has landed, on a shared-memory barrier that nothing completes,
with a short poll limit.  The wait runs out, the CTA records the fault code,
waits (bounded) for its own copies still in flight and returns.  The test
checks that the host reads the code through ``tf_topk_device_fault`` (then
cleared), that the context stays usable, and that the next calls on the
same stream -- the product library's stream plan, whose tickets every launch
clears first, and AUTO -- are exact against the oracle.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_same, device_matrix, to_numpy
from wide_bf16_row_gb300 import synth

pytestmark = pytest.mark.gpu

FAULT_WAIT_TIMEOUT = 1  # the code a wait that ran out records
PLAN_STREAM = 32


def _timeout_library() -> ctypes.CDLL:
    from wide_bf16_row_gb300 import build

    lib = ctypes.CDLL(str(build.build_variant("wait_timeout", ("TF_TOPK_TEST_WAIT_TIMEOUT",))))
    c_i64, c_i32, c_p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    lib.tf_topk_bf16_with_plan.restype = ctypes.c_int
    lib.tf_topk_bf16_with_plan.argtypes = [c_p, c_i64, c_i64, c_i64, c_i32, c_p, c_p, c_p, c_p, c_i32, c_p]
    lib.tf_topk_device_fault.restype = ctypes.c_int
    lib.tf_topk_device_fault.argtypes = []
    return lib


def test_stream_wait_timeout_is_reported_and_the_next_calls_are_exact():
    import torch

    from wide_bf16_row_gb300 import topk

    rows, cols, k = 40, 70000, 20
    x = synth.mixed_rows(rows, cols, seed=5, row_stride=cols, special_frac=0.002, dup_frac=0.01)
    exp = oracle.topk(x, cols, k)
    view, keep = device_matrix(x, cols)
    stream = torch.cuda.current_stream()
    out = (torch.empty((rows, k), dtype=torch.int32, device="cuda"),
           torch.empty((rows, k), dtype=torch.int16, device="cuda"),
           torch.empty((rows,), dtype=torch.int32, device="cuda"),
           torch.empty((rows,), dtype=torch.int32, device="cuda"))

    lib = _timeout_library()
    assert lib.tf_topk_device_fault() == 0
    st = lib.tf_topk_bf16_with_plan(view.data_ptr(), rows, cols, cols, k, out[0].data_ptr(), out[1].data_ptr(),
                                    out[2].data_ptr(), out[3].data_ptr(), PLAN_STREAM, stream.cuda_stream)
    assert st == 0
    torch.cuda.synchronize()  # the kernel returned: no hang, no CUDA error
    assert lib.tf_topk_device_fault() == FAULT_WAIT_TIMEOUT
    assert lib.tf_topk_device_fault() == 0  # reported once, then cleared

    # the context still works, and the product library on the same stream is exact
    assert topk.device_fault() == 0
    for plan in (PLAN_STREAM, 0):
        got = to_numpy(topk.topk_bf16(view, k, plan=plan, stream=stream))
        assert_same(got, exp, f"after a timed-out launch, plan {plan}")
    assert topk.device_fault() == 0

    # the test build again on the same stream: the same code, the same recovery
    st = lib.tf_topk_bf16_with_plan(view.data_ptr(), rows, cols, cols, k, out[0].data_ptr(), out[1].data_ptr(),
                                    out[2].data_ptr(), out[3].data_ptr(), PLAN_STREAM, stream.cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert lib.tf_topk_device_fault() == FAULT_WAIT_TIMEOUT
    del keep
