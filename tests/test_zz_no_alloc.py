"""rowops_online_softmax_noalloc: the split-row online softmax for callers that
cannot allocate device memory (a plugin handed only device pointers, or a
latency-critical path that cannot afford cudaMalloc). Its partials live in a
1 MiB device array owned by the library.

Checked through the C ABI against the oracle (the plain softmax definition in
double precision) at the parity tests' softmax tolerances: the bf16 37 x 50000
case on every element, the fp32 64 x 2^20 outlier workload on sampled rows and
on every row through the closed form of its outlier entries; on two calls in a
row over the array's leftovers, then the first case again; and its size limit,
for an explicit chunk (rejected before any CUDA call) and for the automatic
chunk (rejected after the device lookup, before any launch). Collected last so
that a run stopping at the first failure has already run every other test.
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
def test_noalloc_rejects_oversize_with_automatic_chunk():
    """With chunk 0 the chunk comes from the SM count, so the partial count is
    known only after the device lookup: 131041 rows of 256 columns still need
    more than the array's 131040 partials and are rejected, nothing launched
    (the pointers are fake)."""
    lib = _lib()
    X, Y = 1 << 32, 1 << 40
    assert lib.rowops_online_softmax_noalloc(X, Y, 131041, 256, 256, F32, 0, None) == WORKSPACE


def _check_outlier_rows(x, y):
    """Every row of the +30 outlier workload: its k outlier entries equal
    1 / (k + S), S = sum of exp(x - 30) over the other entries (float64)."""
    hit = x == 30.0
    k = hit.sum(dim=1, dtype=torch.float64)
    S = torch.where(hit, 0.0, torch.exp(x.double() - 30.0)).sum(dim=1)
    want = 1.0 / (k + S)
    got = torch.where(hit, y.double(), 0.0).sum(dim=1) / k
    assert torch.all((got / want - 1).abs() <= 1e-5)
    assert torch.all((y.double().sum(dim=1) - 1).abs() <= 1e-4)


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
def test_noalloc_matches_oracle_twice(oracle):
    """Two calls in a row (different shapes, so the second call runs over the
    first call's leftovers in the shared array) and the first case once more;
    each output against the oracle."""
    from row_wise_reduction_gb300 import workloads
    from tests import gpu_util as gu

    lib = _lib()
    big = workloads.WORKLOADS["online_softmax_f32_64x1048576"]  # 64 x 2^20 fp32, 8192 partials
    small = workloads.Workload("noalloc_bf16", "online_softmax", "bf16", 37, 50000, seed=21, x_std=3.0)

    def run_big():
        x = workloads.make_inputs(big, "cuda")["x"]
        y = torch.full_like(x, float("nan"))
        _call(lib, x, y, 0)
        torch.cuda.synchronize()
        rows = gu.sample_rows(big.M, 4, seed=5)
        ref = oracle.softmax(gu.rows_f32(x, rows))
        C.assert_softmax_close(C.to_f64(y[torch.as_tensor(rows, device=y.device)]), ref, "f32",
                               what="noalloc fp32 64 x 2^20 sampled rows")
        _check_outlier_rows(x, y)

    def run_small():
        x = workloads.make_inputs(small, "cuda")["x"]
        y = torch.full_like(x, float("nan"))
        _call(lib, x, y, 1024)
        torch.cuda.synchronize()
        C.assert_softmax_close(C.to_f64(y), oracle.softmax(gu.rows_f32(x)), "bf16", what="noalloc bf16 37 x 50000")

    run_big()
    run_small()
    run_big()
