"""GPU parity of rowops_bias_residual_gelu (y = GELU(x + b + residual), b per
column) with the oracle, through the C ABI ["Triton Kernel 实现练习" §3.4 Approx
Activation, "fused residual + bias + GELU"].

Tolerances as for LayerNorm+GELU: fp32 max abs 1e-5 (the fp32 sum and the GELU
evaluation err by ~1e-6 at |z| ~ 10), bf16 within one ulp (+1e-5 abs). Both GELU
forms; the 16-byte vector path and the element path (ragged N, strided and
misaligned rows, forced); optional inputs absent; in place on x and on the
residual; guard bands; the full-size bf16 workload on sampled rows.
"""
import numpy as np
import pytest
import torch

from row_wise_reduction_gb300 import rowops_bias_residual_gelu, workloads
from tests import _compare as C
from tests import gpu_util as gu

pytestmark = [pytest.mark.gpu, gu.requires_gpu]

F1 = workloads.WORKLOADS["bias_residual_gelu_f32_4096x768"]
F2 = workloads.WORKLOADS["bias_residual_gelu_bf16_65536x8192"]


def edge(dtype, M, N, seed=31):
    return workloads.Workload(f"brg_{dtype}_{M}x{N}", "bias_residual_gelu", dtype, M, N, seed=seed, affine=True,
                              residual=True)


def host(t):
    return None if t is None else t.float().cpu().numpy()


def place(t: torch.Tensor, ld: int, offset: int):
    M, N = t.shape
    buf = torch.full((M * ld + offset + 8,), float("nan"), dtype=t.dtype, device=t.device)
    view = torch.as_strided(buf, (M, N), (ld, 1), offset)
    view.copy_(t)
    return view


def check(oracle, wl, approximate="none", ld=None, offset=0, use_r=True, use_b=True, inplace=None, rows=None):
    inp = gu.make_x(wl, ld=ld, offset=offset)
    x = inp["x"]
    ldx = x.stride(0) if wl.M > 1 else wl.N
    r = (place(inp["residual"], ldx, offset) if offset else inp["residual"]) if use_r else None
    b = inp["b"] if use_b else None
    xin, rin = gu.rows_f32(x, rows), (gu.rows_f32(r, rows) if r is not None else None)
    buf = inside = None
    if inplace == "x":
        y = x
    elif inplace == "r":
        y = r
    else:
        y, buf, inside = gu.guarded_like(x, offset=offset)
    rowops_bias_residual_gelu(x, r, b, y, approximate)
    torch.cuda.synchronize()
    ref = oracle.bias_residual_gelu(xin, rin, host(b), approximate)
    got = C.to_f64(y if rows is None else y[torch.as_tensor(rows, device=y.device)])
    C.assert_ln_gelu_close(got, ref, wl.dtype, what=f"{wl.name} {approximate}")
    if buf is not None:
        gu.assert_guard_untouched(buf, inside)


@pytest.mark.parametrize("approximate", ["none", "tanh"])
def test_f32_workload_in_full(oracle, approximate):
    check(oracle, F1, approximate)


@pytest.mark.parametrize("approximate", ["none", "tanh"])
def test_bf16_workload_reduced_rows(oracle, approximate):
    check(oracle, F2.with_shape(M=512), approximate)


def test_bf16_workload_full_size_sampled_rows(oracle):
    check(oracle, F2, "none", rows=gu.sample_rows(F2.M, 64, seed=3))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 7, 8, 127, 1000, 4096, 4097, 20000])
def test_widths(oracle, dtype, N):
    check(oracle, edge(dtype, 37, N, seed=N), "none")
    check(oracle, edge(dtype, 37, N, seed=N + 1), "tanh")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_strided_and_misaligned_rows(oracle, dtype):
    for ld, off in [(1040, 0), (1029, 0), (1024, 1), (1032, 3)]:
        check(oracle, edge(dtype, 50, 1024, seed=ld + off), "none", ld=ld, offset=off)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_optional_inputs_and_in_place(oracle, dtype):
    wl = edge(dtype, 64, 2048)
    check(oracle, wl, use_r=False)
    check(oracle, wl, use_b=False)
    check(oracle, wl, use_r=False, use_b=False)
    check(oracle, wl, inplace="x")
    check(oracle, wl, inplace="r")


def test_element_path_forced(oracle, monkeypatch):
    monkeypatch.setenv("ROWOPS_KERNEL", "looped")
    check(oracle, edge("bf16", 40, 4096), "none")
    check(oracle, edge("f32", 40, 768), "tanh")


def test_zero_rows():
    x = torch.empty(0, 64, device="cuda")
    assert rowops_bias_residual_gelu(x).shape == (0, 64)
