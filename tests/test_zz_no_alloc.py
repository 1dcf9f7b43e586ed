"""rowops_online_softmax_noalloc: the split-row online softmax for callers that
cannot allocate device memory (a plugin handed only device pointers, or a
latency-critical path that cannot afford cudaMalloc). Its partials live in a
1 MiB device array owned by the library.

Checked through the C ABI against rowops_online_softmax (the workspace entry
point) with the parity tests' softmax tolerance, on two calls in a row, and
for its size limit. Collected last so that a run stopping at the first
failure has already run every other test.
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from tests import _compare as C

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
F32, BF16 = 0, 1
OK, WORKSPACE = 0, 3


def _lib():
    from row_wise_reduction_gb300 import build
    from row_wise_reduction_gb300.rowops import library

    build.build()
    return library()


def test_noalloc_source_calls_no_allocator():
    """The entry point's translation unit calls no allocating routine."""
    src = open(os.path.join(ROOT, "row_wise_reduction_gb300", "csrc", "online_softmax_noalloc.cu")).read()
    code = re.sub(r"//.*", "", src)
    for name in ("cudaMalloc", "cudaFree", "cudaMallocAsync", "cudaMallocManaged", "malloc(", "new "):
        assert name not in code, name


def test_noalloc_rejects_oversize_and_bad_arguments_before_any_launch():
    lib = _lib()
    f = lib.rowops_online_softmax_noalloc
    X, Y = 1 << 32, 1 << 40  # fake, non-overlapping device addresses: nothing is launched
    # 131041 chunk partials do not fit the 1 MiB array: rejected before any CUDA work
    assert f(X, Y, 131041, 256, 256, F32, 256, None) == WORKSPACE
    assert f(X, Y, 2, 4096, 4096, 9, 0, None) == 1
    assert f(X, Y, 2, 4096, 4000, F32, 0, None) == 1
    assert f(X, Y, 2, 4096, 4096, F32, 100, None) == 1
    assert f(None, None, 0, 4096, 4096, F32, 0, None) == OK


def _call(lib, x, y, chunk):
    M, N = x.shape
    st = lib.rowops_online_softmax_noalloc(x.data_ptr(), y.data_ptr(), M, N, x.stride(0), F32 if x.dtype == torch.float32
                                           else BF16, chunk, torch.cuda.current_stream().cuda_stream)
    assert st == OK, st


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
def test_noalloc_matches_workspace_entry_point_twice():
    """Two calls in a row (different shapes, so the second call runs over the
    first call's leftovers in the shared array); each matches
    rowops_online_softmax on the same input within the softmax tolerance."""
    from row_wise_reduction_gb300 import rowops_online_softmax, workloads

    lib = _lib()
    cases = [
        (workloads.WORKLOADS["online_softmax_f32_64x1048576"].with_shape(M=64), 0),  # 64 x 2^20, 8192 partials
        (workloads.Workload("noalloc_bf16", "online_softmax", "bf16", 37, 50000, seed=21, x_std=3.0), 1024),
    ]
    for wl, chunk in cases:
        x = workloads.make_inputs(wl, "cuda")["x"]
        want = rowops_online_softmax(x, chunk=chunk)
        got = torch.full_like(x, float("nan"))
        _call(lib, x, got, chunk)
        torch.cuda.synchronize()
        C.assert_softmax_close(C.to_f64(got), C.to_f64(want), wl.dtype, what=f"noalloc {wl.name}")
        assert torch.isfinite(got).all()
    # and the first case once more, after the second case used the array
    wl, chunk = cases[0]
    x = workloads.make_inputs(wl, "cuda")["x"]
    want = rowops_online_softmax(x, chunk=chunk)
    got = torch.empty_like(x)
    _call(lib, x, got, chunk)
    torch.cuda.synchronize()
    C.assert_softmax_close(C.to_f64(got), C.to_f64(want), "f32", what="noalloc repeat")
