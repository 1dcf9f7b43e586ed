"""GPU parity of rowops_row_sum and rowops_row_max with the oracle, through the
C ABI ["Triton Kernel 实现练习" §2.2 Row-wise Sum, §2.3 Row-wise Max].

Row sums: within 1e-5 * sum_j |x_ij| of the oracle's double sum (fp32
accumulation over at most a few thousand terms per thread); row maxima: equal
to the oracle bit for bit (the maximum is one of the inputs, exact in fp32),
NaN rows NaN. Ragged, strided and misaligned rows, special values, every
kernel family, the full-size bf16 workloads on every row.
"""
import numpy as np
import pytest
import torch

from row_wise_reduction_gb300 import rowops_device_status, rowops_row_max, rowops_row_sum, workloads
from tests import gpu_util as gu

pytestmark = [pytest.mark.gpu, gu.requires_gpu]


def wl_of(dtype, M, N, seed=3, std=2.0):
    return workloads.Workload(f"red_{dtype}_{M}x{N}", "row_sum", dtype, M, N, seed=seed, x_std=std)


def check_sum(oracle, x):
    got = rowops_row_sum(x)
    torch.cuda.synchronize()
    xin = gu.rows_f32(x)
    ref = oracle.row_sum(xin)
    scale = np.abs(xin.astype(np.float64)).sum(axis=1)
    g = got.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isnan(g), np.isnan(ref)) and np.array_equal(g[~fin & ~np.isnan(ref)], ref[~fin & ~np.isnan(ref)])
    assert np.all(np.abs(g[fin] - ref[fin]) <= 1e-5 * scale[fin] + 1e-30), np.max(np.abs(g[fin] - ref[fin]) - 1e-5 * scale[fin])
    assert rowops_device_status() == 0


def check_max(oracle, x):
    got = rowops_row_max(x)
    torch.cuda.synchronize()
    ref = oracle.row_max(gu.rows_f32(x))
    np.testing.assert_array_equal(got.cpu().numpy().astype(np.float64), ref)
    assert rowops_device_status() == 0


RAGGED_N = [1, 2, 3, 7, 8, 9, 17, 127, 128, 129, 511, 512, 513, 767, 768, 4095, 4096, 4097, 8192, 16385, 32768,
            32769, 100003]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", RAGGED_N)
def test_row_reductions_ragged(oracle, dtype, N):
    x = gu.make_x(wl_of(dtype, 23 if N < 50000 else 5, N, seed=N))["x"]
    check_sum(oracle, x)
    check_max(oracle, x)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,ld,offset", [(127, 127, 1), (4097, 4097, 0), (4096, 4100, 3), (768, 780, 0),
                                         (8192, 8192, 1), (40000, 40003, 1)])
def test_row_reductions_strided_misaligned(oracle, dtype, N, ld, offset):
    x = gu.make_x(wl_of(dtype, 19, N, seed=ld), ld=ld, offset=offset)["x"]
    check_sum(oracle, x)
    check_max(oracle, x)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [100, 4096])
def test_row_reductions_special_values(oracle, dtype, N):
    x = gu.make_x(wl_of(dtype, 6, N, seed=1))["x"]
    x[1] = float("-inf")
    x[2, N // 3] = float("nan")
    x[3, N - 1] = float("inf")
    x[4, 0] = float("-inf")
    x[5] = 0
    check_sum(oracle, x)
    check_max(oracle, x)
    m = rowops_row_max(x).cpu()
    assert m[1] == float("-inf") and torch.isnan(m[2]) and m[3] == float("inf")


@pytest.mark.parametrize("env", [{"ROWOPS_KERNEL": "tma"}, {"ROWOPS_KERNEL": "reg"}, {"ROWOPS_KERNEL": "looped"},
                                 {"ROWOPS_KERNEL": "tma", "ROWOPS_RING_BUFFERS": "4"},
                                 {"ROWOPS_KERNEL": "tma", "ROWOPS_FORCE_TPR": "512", "ROWOPS_FORCE_VPT": "2"},
                                 {"ROWOPS_KERNEL": "reg", "ROWOPS_FORCE_TPR": "1024", "ROWOPS_FORCE_VPT": "1"}],
                         ids=lambda e: ",".join(f"{k[7:]}={v}" for k, v in e.items()))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1000, 4096, 4097])
def test_row_reductions_every_family(oracle, monkeypatch, env, dtype, N):
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    x = gu.make_x(wl_of(dtype, 301, N, seed=N + 1))["x"]
    check_sum(oracle, x)
    check_max(oracle, x)


@pytest.mark.parametrize("name", ["row_sum_bf16_65536x8192", "row_max_bf16_65536x8192"])
def test_row_reductions_full_size(oracle, name):
    """Every row of the bf16 65536 x 8192 workloads: sums against torch's float64
    sum within the stated tolerance, maxima equal to torch's; 16 sampled rows
    against the oracle."""
    wl = workloads.WORKLOADS[name]
    x = gu.make_x(wl)["x"]
    if wl.op == "row_sum":
        got = rowops_row_sum(x).double()
        ref = x.double().sum(dim=1)
        assert torch.all((got - ref).abs() <= 1e-5 * x.double().abs().sum(dim=1))
    else:
        got = rowops_row_max(x)
        assert torch.equal(got, x.float().amax(dim=1))
    rows = gu.sample_rows(wl.M, 16, seed=5)
    sub = x[torch.as_tensor(rows, device=x.device)]
    check_sum(oracle, sub)
    check_max(oracle, sub)


def test_row_reductions_empty_and_out_buffer(oracle):
    x = torch.empty(0, 64, device="cuda")
    assert rowops_row_sum(x).shape == (0,)
    x = gu.make_x(wl_of("f32", 8, 64))["x"]
    out = torch.full((8,), 7.0, device="cuda")
    assert rowops_row_max(x, out) is out
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy().astype(np.float64), oracle.row_max(gu.rows_f32(x)))
