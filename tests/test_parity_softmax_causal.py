"""GPU parity of rowops_softmax_causal with the oracle, through the C ABI
["Triton Kernel 实现练习" §5.1 causal mask, §2.4 softmax].

Row r keeps the columns c <= (r mod period) + offset; the masked columns are
never read. Checks: the oracle on every element at reduced sizes and on
sampled rows of the full causal workload (bf16 32768 x 4096, period 4096);
masked outputs exactly 0 and rows summing to 1 on every row; NaN written into
the masked region changes nothing; on the workload's input (-inf in the masked
columns) the causal kernel equals rowops_softmax bit for bit. Edge cases:
ragged and strided rows, periods and offsets that keep nothing or everything,
both kernel families, ring depths and tiles, in place, guard bands.
"""
import numpy as np
import pytest
import torch

from row_wise_reduction_gb300 import rowops_device_status, rowops_softmax, rowops_softmax_causal, workloads
from tests import _compare as C
from tests import gpu_util as gu

pytestmark = [pytest.mark.gpu, gu.requires_gpu]

W3 = workloads.WORKLOADS["softmax_bf16_causal_32768x4096"]


def rows_kept(M, N, period, offset):
    r = np.arange(M)
    return np.clip(r % period + offset + 1, 0, N)


def plain(dtype, M, N, seed=7, std=2.0):
    """Unmasked random rows (the causal call does the masking)."""
    return workloads.Workload(f"causal_{dtype}_{M}x{N}", "softmax", dtype, M, N, seed=seed, x_std=std)


def poison_masked(x, period, offset, value=float("nan")):
    M, N = x.shape
    kept = torch.as_tensor(rows_kept(M, N, period, offset), device=x.device)
    mask = torch.arange(N, device=x.device)[None, :] >= kept[:, None]
    x.masked_fill_(mask, value)
    return mask


def check(oracle, wl, period, offset, ld=None, offset_el=0, inplace=False, poison=True):
    inp = gu.make_x(wl, ld=ld, offset=offset_el)
    x = inp["x"]
    xin = gu.rows_f32(x)  # before poisoning: the oracle never reads the masked entries either
    if poison:
        poison_masked(x, period, offset)
    if inplace:
        y, buf, inside = x, None, None
    else:
        y, buf, inside = gu.guarded_like(x, offset=offset_el)
    rowops_softmax_causal(x, period, offset, y)
    torch.cuda.synchronize()
    ref = oracle.softmax_causal(xin, period, offset)
    C.assert_softmax_close(C.to_f64(y), ref, wl.dtype, what=f"{wl.name} period={period} offset={offset}")
    if buf is not None:
        gu.assert_guard_untouched(buf, inside)
    assert rowops_device_status() == 0
    return y


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,period,offset", [(300, 4096, 4096, 0), (300, 4096, 128, 0), (257, 8192, 100, 37),
                                               (64, 2048, 64, -3), (100, 1024, 7, 1000), (50, 4096, 4096, -1)])
def test_causal_full_rows(oracle, dtype, M, N, period, offset):
    check(oracle, plain(dtype, M, N, seed=M + N), period, offset)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 5, 127, 768, 4097, 16385, 40000])
def test_causal_ragged_rows(oracle, dtype, N):
    check(oracle, plain(dtype, 37, N, seed=N), period=37, offset=N // 3)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,ld,offset_el", [(4096, 4100, 0), (4096, 4096, 1), (1000, 1003, 2)])
def test_causal_strided_and_misaligned(oracle, dtype, N, ld, offset_el):
    check(oracle, plain(dtype, 41, N, seed=ld), period=41, offset=5, ld=ld, offset_el=offset_el)


@pytest.mark.parametrize("env", [{"ROWOPS_KERNEL": "looped"}, {"ROWOPS_RING_BUFFERS": "4"},
                                 {"ROWOPS_FORCE_TPR": "128", "ROWOPS_FORCE_VPT": "4"}],
                         ids=lambda e: ",".join(f"{k[7:]}={v}" for k, v in e.items()))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_causal_kernel_variants(oracle, monkeypatch, env, dtype):
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    check(oracle, plain(dtype, 517, 4096, seed=5), period=4096, offset=0)
    check(oracle, plain(dtype, 3, 4096, seed=6), period=2, offset=7)


def test_causal_in_place(oracle):
    check(oracle, plain("bf16", 200, 4096), period=4096, offset=0, inplace=True)


def test_causal_workload_full_size(oracle, monkeypatch):
    """bf16 32768 x 4096 with the workload's causal pattern: the default
    launch; 48 sampled rows against the oracle, on every row masked outputs
    exactly 0 and the kept outputs summing to 1; within the softmax tolerance
    of rowops_softmax on the same input (which reads the -inf masked entries),
    and equal to it bit for bit when both run the same tile."""
    inp = gu.make_x(W3)
    x = inp["x"]
    y = rowops_softmax_causal(x, 4096, 0)
    y_plain = rowops_softmax(x)
    torch.cuda.synchronize()
    C.assert_softmax_close(C.to_f64(y), C.to_f64(y_plain), "bf16")
    monkeypatch.setenv("ROWOPS_FORCE_TPR", "128")
    monkeypatch.setenv("ROWOPS_FORCE_VPT", "4")
    assert torch.equal(rowops_softmax_causal(x, 4096, 0).view(torch.int16), rowops_softmax(x).view(torch.int16))
    monkeypatch.delenv("ROWOPS_FORCE_TPR")
    monkeypatch.delenv("ROWOPS_FORCE_VPT")
    kept = torch.as_tensor(rows_kept(W3.M, W3.N, 4096, 0), device=x.device)
    masked = torch.arange(W3.N, device=x.device)[None, :] >= kept[:, None]
    assert torch.count_nonzero(y[masked]) == 0
    sums = y.double().sum(dim=1)
    assert torch.all((sums - 1).abs() <= 4e-3)  # bf16 outputs: each within 2^-9 relative
    rows = gu.sample_rows(W3.M, 48, seed=3)
    ref = np.stack([oracle.softmax_causal_rows_at(gu.rows_f32(x, [r])[0], r, 4096, 0) for r in rows])
    C.assert_softmax_close(C.to_f64(y[torch.as_tensor(rows, device=y.device)]), ref, "bf16")
    # NaN in the masked region: never read, same output
    x.masked_fill_(masked, float("nan"))
    y2 = rowops_softmax_causal(x, 4096, 0)
    torch.cuda.synchronize()
    assert torch.equal(y2.view(torch.int16), y.view(torch.int16))
    assert rowops_device_status() == 0


def test_causal_empty_is_noop():
    x = torch.empty(0, 4096, device="cuda", dtype=torch.bfloat16)
    assert rowops_softmax_causal(x).shape == (0, 4096)
