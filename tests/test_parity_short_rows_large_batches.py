"""GPU parity, through the C ABI, of the default kernel choice on batches above
32 MiB of rows shorter than the row pipeline's crossover (they take the
register-resident kernels, or for LayerNorm+GELU rows of at most 256 columns
the chunked kernel): softmax, LayerNorm+GELU, RMSNorm, row sum and row max on
sampled rows against the oracle, every row finite; and the rows just at each
crossover, which keep the row pipeline.
"""
import numpy as np
import pytest
import torch

from row_wise_reduction_gb300 import (rowops_device_status, rowops_layernorm_gelu, rowops_rmsnorm, rowops_row_max,
                                      rowops_row_sum, rowops_softmax, workloads)
from tests import _compare as C
from tests import gpu_util as gu

pytestmark = [pytest.mark.gpu, gu.requires_gpu]

SHAPES = [("f32", 262144, 256), ("bf16", 262144, 512), ("f32", 131072, 512), ("bf16", 131072, 1024),
          ("f32", 65536, 2048), ("bf16", 65536, 2048), ("bf16", 65536, 4096)]


def wl(op, dtype, M, N):
    return workloads.Workload(f"short_{op}_{dtype}_{M}x{N}", op, dtype, M, N, seed=M % 97 + N, affine=True)


def host(t):
    return None if t is None else t.float().cpu().numpy()


@pytest.mark.parametrize("dtype,M,N", SHAPES)
def test_softmax_large_batches(oracle, dtype, M, N):
    x = gu.make_x(wl("softmax", dtype, M, N))["x"]
    y = rowops_softmax(x)
    torch.cuda.synchronize()
    rows = gu.sample_rows(M, 24, seed=N)
    C.assert_softmax_close(C.to_f64(y[torch.as_tensor(rows, device=y.device)]), oracle.softmax(gu.rows_f32(x, rows)),
                           dtype)
    assert torch.isfinite(y).all()
    assert rowops_device_status() == 0


@pytest.mark.parametrize("dtype,M,N", SHAPES + [("f32", 131072, 256)])
def test_layernorm_gelu_large_batches(oracle, dtype, M, N):
    inp = gu.make_x(wl("layernorm_gelu", dtype, M, N))
    x, w, b = inp["x"], inp["w"], inp["b"]
    y = rowops_layernorm_gelu(x, w, b, 1e-5)
    torch.cuda.synchronize()
    rows = gu.sample_rows(M, 24, seed=N)
    ref = oracle.layernorm_gelu(gu.rows_f32(x, rows), host(w), host(b), 1e-5)
    C.assert_ln_gelu_close(C.to_f64(y[torch.as_tensor(rows, device=y.device)]), ref, dtype)
    assert torch.isfinite(y).all()
    assert rowops_device_status() == 0


@pytest.mark.parametrize("dtype,M,N", SHAPES)
def test_rmsnorm_large_batches(oracle, dtype, M, N):
    inp = gu.make_x(wl("rmsnorm", dtype, M, N))
    x, w = inp["x"], inp["w"]
    y = rowops_rmsnorm(x, w, 1e-5)
    torch.cuda.synchronize()
    rows = gu.sample_rows(M, 24, seed=N)
    C.assert_rms_close(C.to_f64(y[torch.as_tensor(rows, device=y.device)]),
                       oracle.rmsnorm(gu.rows_f32(x, rows), host(w), 1e-5), dtype)
    assert torch.isfinite(y).all()
    assert rowops_device_status() == 0


@pytest.mark.parametrize("dtype,M,N", SHAPES + [("bf16", 32768, 8192)])
def test_row_sum_and_max_large_batches(oracle, dtype, M, N):
    x = gu.make_x(wl("row_sum", dtype, M, N))["x"]
    s, m = rowops_row_sum(x), rowops_row_max(x)
    torch.cuda.synchronize()
    xin = gu.rows_f32(x)  # every row
    ref = oracle.row_sum(xin)
    scale = np.abs(xin.astype(np.float64)).sum(axis=1)
    assert np.all(np.abs(s.cpu().numpy().astype(np.float64) - ref) <= 1e-5 * scale + 1e-30)
    np.testing.assert_array_equal(m.cpu().numpy().astype(np.float64), oracle.row_max(xin))
    assert rowops_device_status() == 0
