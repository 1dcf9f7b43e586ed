"""GPU parity of rowops_rmsnorm and rowops_fused_residual_rmsnorm with the
oracle, through the C ABI ["Triton Kernel 实现练习" §4.2, §4.3].

y is compared with the oracle's double result within the stated tolerance;
residual_out must equal the oracle's x + residual rounded to the I/O type bit
for bit (one correctly rounded addition). Workloads: fp32 4096 x 768 in full,
bf16 65536 x 8192 on reduced rows in full and at full size on sampled rows;
edge cases: ragged and strided rows, every 16-byte phase class, pointers at
different offsets modulo 16 bytes, in place, NULL weight, zero rows, every
kernel family and tile, guard bands around both outputs.
"""
import numpy as np
import pytest
import torch

from row_wise_reduction_gb300 import rowops_device_status, rowops_fused_residual_rmsnorm, rowops_rmsnorm, workloads
from tests import _compare as C
from tests import gpu_util as gu

pytestmark = [pytest.mark.gpu, gu.requires_gpu]

R1 = workloads.WORKLOADS["rmsnorm_f32_4096x768"]
R2 = workloads.WORKLOADS["rmsnorm_bf16_65536x8192"]
F1 = workloads.WORKLOADS["residual_rmsnorm_f32_4096x768"]
F2 = workloads.WORKLOADS["residual_rmsnorm_bf16_65536x8192"]


def edge(op, dtype, M, N, seed=11):
    return workloads.Workload(f"edge_{op}_{dtype}_{M}x{N}", op, dtype, M, N, seed=seed, affine=True,
                              residual=(op == "residual_rmsnorm"))


def host(t):
    return None if t is None else t.float().cpu().numpy()


def place(t: torch.Tensor, ld: int, offset: int):
    """A copy of the (M, N) tensor ``t`` as a view of row stride ``ld`` starting
    ``offset`` elements into a NaN-filled buffer."""
    M, N = t.shape
    buf = torch.full((M * ld + offset + 8,), float("nan"), dtype=t.dtype, device=t.device)
    view = torch.as_strided(buf, (M, N), (ld, 1), offset)
    view.copy_(t)
    return view


def check_rms(oracle, wl, ld=None, offset=0, yoffset=None, inplace=False, use_w=True):
    inp = gu.make_x(wl, ld=ld, offset=offset)
    x = inp["x"]
    w = inp.get("w") if use_w else None
    xin = gu.rows_f32(x)
    if inplace:
        y, buf, inside = x, None, None
    else:
        y, buf, inside = gu.guarded_like(x, offset=offset if yoffset is None else yoffset)
    rowops_rmsnorm(x, w, wl.eps, y)
    torch.cuda.synchronize()
    C.assert_rms_close(C.to_f64(y), oracle.rmsnorm(xin, host(w), wl.eps), wl.dtype, what=wl.name)
    if buf is not None:
        gu.assert_guard_untouched(buf, inside)
    assert rowops_device_status() == 0


def check_res(oracle, wl, ld=None, offsets=(0, 0, 0, 0), alias=None, use_w=True):
    """offsets of x, residual, y, residual_out (elements); alias: None, "ro=r",
    "ro=x", "y=x", "y=x,ro=r", "y=r,ro=x"."""
    ld = wl.N if ld is None else ld
    inp = gu.make_x(wl, ld=ld, offset=offsets[0])
    x = inp["x"]
    r = place(inp["residual"], ld, offsets[1]) if offsets[1] else inp["residual"]
    w = inp.get("w") if use_w else None
    xin, rin = gu.rows_f32(x), gu.rows_f32(r)
    guards = []
    alias = alias or ""
    if "y=x" in alias:
        y = x
    elif "y=r" in alias:
        y = r
    else:
        y, buf, inside = gu.guarded_like(x, offset=offsets[2])
        guards.append((buf, inside))
    if "ro=r" in alias:
        ro = r
    elif "ro=x" in alias:
        ro = x
    else:
        ro, buf, inside = gu.guarded_like(x, offset=offsets[3])
        guards.append((buf, inside))
    rowops_fused_residual_rmsnorm(x, r, w, wl.eps, y, ro)
    torch.cuda.synchronize()
    s_ref, y_ref = oracle.residual_rmsnorm(xin, rin, host(w), wl.eps, wl.dtype)
    np.testing.assert_array_equal(C.to_f64(ro), s_ref, err_msg=f"{wl.name}: residual_out")
    C.assert_rms_close(C.to_f64(y), y_ref, wl.dtype, what=wl.name)
    for buf, inside in guards:
        gu.assert_guard_untouched(buf, inside)
    assert rowops_device_status() == 0


def test_rmsnorm_f32_4096x768_full(oracle):
    check_rms(oracle, R1)


def test_residual_rmsnorm_f32_4096x768_full(oracle):
    check_res(oracle, F1)


def test_rmsnorm_bf16_reduced_rows(oracle):
    check_rms(oracle, R2.with_shape(M=1000))


def test_residual_rmsnorm_bf16_reduced_rows(oracle):
    check_res(oracle, F2.with_shape(M=1000))


@pytest.mark.parametrize("wl", [R2, F2], ids=lambda w: w.name)
def test_bf16_full_size_sampled(oracle, wl):
    """Full-size bf16 workloads (65536 x 8192) in the default launch
    configuration: 48 sampled rows against the oracle; residual_out equal to
    x + residual rounded to bf16 on every element (torch's own bf16 add)."""
    inp = gu.make_x(wl)
    x, w = inp["x"], inp["w"]
    rows = gu.sample_rows(wl.M, 48, seed=wl.N)
    idx = torch.as_tensor(rows, device=x.device)
    if wl.op == "rmsnorm":
        y = rowops_rmsnorm(x, w, wl.eps)
        torch.cuda.synchronize()
        ref = oracle.rmsnorm(gu.rows_f32(x, rows), host(w), wl.eps)
    else:
        r = inp["residual"]
        y, ro = rowops_fused_residual_rmsnorm(x, r, w, wl.eps)
        torch.cuda.synchronize()
        assert torch.equal(ro, x + r)
        s_ref, ref = oracle.residual_rmsnorm(gu.rows_f32(x, rows), gu.rows_f32(r, rows), host(w), wl.eps, "bf16")
        np.testing.assert_array_equal(C.to_f64(ro[idx]), s_ref)
    C.assert_rms_close(C.to_f64(y[idx]), ref, "bf16", what=wl.name)
    assert torch.isfinite(y).all()
    assert rowops_device_status() == 0


RAGGED_N = [1, 2, 3, 5, 8, 9, 17, 31, 127, 128, 129, 767, 768, 769, 4095, 4097, 8192, 12288, 16385, 20000,
            32769, 40000]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", RAGGED_N)
def test_rmsnorm_ragged_n(oracle, dtype, N):
    check_rms(oracle, edge("rmsnorm", dtype, 23, N, seed=N))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", RAGGED_N)
def test_residual_rmsnorm_ragged_n(oracle, dtype, N):
    check_res(oracle, edge("residual_rmsnorm", dtype, 23, N, seed=N))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,ld,offset", [(127, 127, 1), (4097, 4097, 0), (4097, 4105, 3), (768, 780, 0),
                                         (8192, 8192, 1), (40000, 40003, 1)])
def test_strided_and_misaligned_rows(oracle, dtype, N, ld, offset):
    check_rms(oracle, edge("rmsnorm", dtype, 19, N, seed=ld), ld=ld, offset=offset)
    check_res(oracle, edge("residual_rmsnorm", dtype, 19, N, seed=ld), ld=ld, offsets=(offset,) * 4)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [768, 8192])
def test_pointers_out_of_phase(oracle, dtype, N):
    """Rows of the tensors at different offsets modulo 16 bytes (the looped form)."""
    check_rms(oracle, edge("rmsnorm", dtype, 9, N), offset=1, yoffset=0)
    wl = edge("residual_rmsnorm", dtype, 9, N)
    for offs in [(0, 1, 0, 0), (0, 0, 1, 0), (0, 0, 0, 3), (2, 1, 0, 3)]:
        check_res(oracle, wl, offsets=offs)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [127, 768, 8192, 4097])
@pytest.mark.parametrize("alias", ["ro=r", "ro=x", "y=x", "y=x,ro=r", "y=r,ro=x"])
def test_residual_in_place(oracle, dtype, N, alias):
    check_res(oracle, edge("residual_rmsnorm", dtype, 37, N, seed=N + 1), alias=alias)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [127, 8192])
def test_rmsnorm_in_place_and_null_weight(oracle, dtype, N):
    check_rms(oracle, edge("rmsnorm", dtype, 29, N), inplace=True)
    check_rms(oracle, edge("rmsnorm", dtype, 29, N), use_w=False)
    check_res(oracle, edge("residual_rmsnorm", dtype, 29, N), use_w=False)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [64, 4096, 4097])
def test_zero_rows(oracle, dtype, N):
    """All-zero rows give rsqrt(eps) * 0 = 0 (no NaN), as do x = -residual."""
    dt = workloads.torch_dtype(dtype)
    x = torch.zeros(6, N, dtype=dt, device="cuda")
    x[3] = 1.5
    y = rowops_rmsnorm(x)
    torch.cuda.synchronize()
    C.assert_rms_close(C.to_f64(y), oracle.rmsnorm(gu.rows_f32(x), None, 1e-5), dtype)
    r = -x
    y2, ro = rowops_fused_residual_rmsnorm(x, r)
    torch.cuda.synchronize()
    assert torch.count_nonzero(ro) == 0 and torch.count_nonzero(y2) == 0


FAMILIES = [{"ROWOPS_KERNEL": "reg"}, {"ROWOPS_KERNEL": "looped"}, {"ROWOPS_KERNEL": "tma"},
            {"ROWOPS_KERNEL": "tma", "ROWOPS_ROWS_PER_CTA": "1"}, {"ROWOPS_KERNEL": "tma", "ROWOPS_ROWS_PER_CTA": "2"},
            {"ROWOPS_KERNEL": "tma", "ROWOPS_ROWS_PER_CTA": "4"}, {"ROWOPS_KERNEL": "tma", "ROWOPS_ROWS_PER_CTA": "8"},
            {"ROWOPS_KERNEL": "tma", "ROWOPS_RING_BUFFERS": "3"},
            {"ROWOPS_KERNEL": "tma", "ROWOPS_FORCE_TPR": "128", "ROWOPS_FORCE_VPT": "8"},
            {"ROWOPS_KERNEL": "tma", "ROWOPS_FORCE_TPR": "512", "ROWOPS_FORCE_VPT": "2"},
            {"ROWOPS_KERNEL": "tma", "ROWOPS_FORCE_TPR": "64", "ROWOPS_FORCE_VPT": "1"},
            {"ROWOPS_KERNEL": "tma", "ROWOPS_SCHED": "static"},
            {"ROWOPS_KERNEL": "tma", "ROWOPS_SCHED": "dynamic", "ROWOPS_UNIT_ROWS": "3"},
            {"ROWOPS_KERNEL": "tma", "ROWOPS_SCHED": "dynamic", "ROWOPS_ROWS_PER_CTA": "8", "ROWOPS_RING_BUFFERS": "2"}]


@pytest.mark.parametrize("env", FAMILIES, ids=lambda e: ",".join(f"{k[7:]}={v}" for k, v in e.items()))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [256, 768, 4096, 4097, 8192, 8193])
def test_every_kernel_family(oracle, monkeypatch, env, dtype, N):
    """Forced kernel families, row groups per CTA, ring depths and tiles
    (combinations a kernel cannot take fall back to the next family and are
    then checked there); 157 rows span several CTAs and every phase class."""
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    check_rms(oracle, edge("rmsnorm", dtype, 157, N, seed=N + 5))
    check_res(oracle, edge("residual_rmsnorm", dtype, 157, N, seed=N + 6))


@pytest.mark.parametrize("M", [1, 3, 9])
def test_fewer_rows_than_phase_classes(oracle, monkeypatch, M):
    monkeypatch.setenv("ROWOPS_KERNEL", "tma")
    check_rms(oracle, edge("rmsnorm", "bf16", M, 4097, seed=M))
    check_res(oracle, edge("residual_rmsnorm", "bf16", M, 4097, seed=M))


def test_deterministic():
    wl = edge("residual_rmsnorm", "bf16", 300, 8192)
    inp = gu.make_x(wl)
    a, ra = rowops_fused_residual_rmsnorm(inp["x"], inp["residual"], inp["w"])
    b, rb = rowops_fused_residual_rmsnorm(inp["x"], inp["residual"], inp["w"])
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16)) and torch.equal(ra, rb)


def test_empty_is_noop():
    x = torch.empty(0, 4096, device="cuda")
    assert rowops_rmsnorm(x).shape == (0, 4096)
    y, ro = rowops_fused_residual_rmsnorm(x, x.clone())
    assert y.shape == (0, 4096) and ro.shape == (0, 4096)
