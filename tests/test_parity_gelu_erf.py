"""GPU parity of rowops_layernorm_gelu_erf (LayerNorm -> affine -> exact GELU)
and rowops_gelu (elementwise, exact and tanh forms) with the oracle, through
the C ABI ["Triton Kernel 实现练习" §3.4 Approx Activation, §4.1 LayerNorm].
Tolerances as for LayerNorm+GELU: fp32 max abs 1e-5, bf16 1 ulp (+1e-5 abs,
as there). Kernel families, ragged and strided rows, tails of the GELU.
"""
import numpy as np
import pytest
import torch

from row_wise_reduction_gb300 import rowops_device_status, rowops_gelu, rowops_layernorm_gelu_erf, workloads
from tests import _compare as C
from tests import gpu_util as gu

pytestmark = [pytest.mark.gpu, gu.requires_gpu]


def edge(dtype, M, N, seed=11):
    return workloads.Workload(f"erf_{dtype}_{M}x{N}", "layernorm_gelu_erf", dtype, M, N, seed=seed, affine=True)


def check_ln(oracle, wl, ld=None, offset=0):
    inp = gu.make_x(wl, ld=ld, offset=offset)
    x, w, b = inp["x"], inp["w"], inp["b"]
    y, buf, inside = gu.guarded_like(x, offset=offset)
    rowops_layernorm_gelu_erf(x, w, b, wl.eps, y)
    torch.cuda.synchronize()
    ref = oracle.layernorm_gelu_erf(gu.rows_f32(x), w.float().cpu().numpy(), b.float().cpu().numpy(), wl.eps)
    C.assert_ln_gelu_close(C.to_f64(y), ref, wl.dtype, what=wl.name)
    gu.assert_guard_untouched(buf, inside)
    assert rowops_device_status() == 0


def test_ln_gelu_erf_f32_4096x768(oracle):
    check_ln(oracle, workloads.WORKLOADS["layernorm_gelu_erf_f32_4096x768"])


def test_ln_gelu_erf_bf16_reduced_rows(oracle):
    check_ln(oracle, workloads.WORKLOADS["layernorm_gelu_erf_bf16_65536x8192"].with_shape(M=1000))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 5, 127, 768, 4096, 4097, 8192, 16385, 40000])
def test_ln_gelu_erf_ragged(oracle, dtype, N):
    check_ln(oracle, edge(dtype, 23, N, seed=N))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 33, 127, 200, 256])
@pytest.mark.parametrize("M", [5, 1001])
def test_ln_gelu_erf_flat_chunks(oracle, monkeypatch, dtype, N, M):
    """The exact form of the kernel for short back-to-back rows by chunks of
    rows (forced)."""
    monkeypatch.setenv("ROWOPS_KERNEL", "flat")
    check_ln(oracle, edge(dtype, M, N, seed=N + M))


@pytest.mark.parametrize("env", [{"ROWOPS_KERNEL": "tma"}, {"ROWOPS_KERNEL": "reg"}, {"ROWOPS_KERNEL": "looped"},
                                 {"ROWOPS_KERNEL": "tma", "ROWOPS_ROWS_PER_CTA": "1"},
                                 {"ROWOPS_KERNEL": "tma", "ROWOPS_ROWS_PER_CTA": "4"}],
                         ids=lambda e: ",".join(f"{k[7:]}={v}" for k, v in e.items()))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [768, 4096, 4097])
def test_ln_gelu_erf_every_family(oracle, monkeypatch, env, dtype, N):
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    check_ln(oracle, edge(dtype, 157, N, seed=N + 3))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("approximate", ["none", "tanh"])
@pytest.mark.parametrize("n,offset", [(1, 0), (7, 0), (1000, 0), (1000, 1), (1 << 20, 0), (1000003, 3)])
def test_elementwise_gelu(oracle, dtype, approximate, n, offset):
    """x spread over [-12, 12] plus N(0, 1) values; the exact form's negative
    tail (|y| ~ 1e-32 at x = -12) is within the bf16 ulp or the fp32 1e-5."""
    dt = workloads.torch_dtype(dtype)
    g = torch.Generator(device="cuda").manual_seed(n)
    base = torch.full((n + offset,), float("nan"), device="cuda", dtype=dt)
    x = base[offset:]
    x.copy_((torch.linspace(-12, 12, n, device="cuda") + torch.randn(n, device="cuda", generator=g)).to(dt))
    y = rowops_gelu(x, approximate=approximate)
    torch.cuda.synchronize()
    xin = x.float().cpu().numpy().astype(np.float64)
    ref = oracle.gelu_erf(xin) if approximate == "none" else oracle.gelu_tanh(xin)
    C.assert_ln_gelu_close(C.to_f64(y), ref, dtype, what=f"gelu {approximate}")
    if dtype == "f32":
        # error bounds from the arithmetic: both forms take 2^arg of an fp32 argument whose rounding
        # (~|arg| 2^-23) becomes that much relative error of the result, arg = |x| (2.31 + 0.103 x^2)
        # for the tanh form and -log2(e) P(x) ~ |x| (2.31 + 0.105 x^2) for the exact form's fitted
        # odd polynomial P, which adds its own 7e-8 (the form's distance from x Phi(x)); the
        # approximate exp2 / reciprocal add a few ulps, relative to the result. The oracle's tanh form
        # evaluates 1 + tanh(v) as printed, which cancels in double for v < -19, so its own error
        # there, ~2^-53 |x|, is added as a floor.
        err = np.abs(C.to_f64(y) - ref)
        arg = np.abs(xin) * (2.31 + (0.103 if approximate == "tanh" else 0.105) * xin**2)
        bound = (1.0 + arg) * 5e-7 * np.abs(ref) + 2.0**-50 * np.abs(xin) + 1e-37
        if approximate == "none":
            bound = bound + 7e-8
        assert np.all(err <= bound), float(np.max(err - bound))
    # in place
    x2 = x.clone()
    rowops_gelu(x2, x2, approximate=approximate)
    torch.cuda.synchronize()
    assert torch.equal(x2, y)
