"""GPU parity of rowops_layernorm_gelu_backward with the oracle, through the C
ABI ["PyTorch 自定义 CUDA 算子与 Triton 编程" §三 FusedLayerNormGELU: the exact
gradient of LayerNorm -> affine -> tanh-GELU].

Tolerances (derived from fp32 arithmetic, u = 2^-24):
- dx: every element within 1e-5 S of the oracle's double value, S = rstd (|dxh|
  + mean |dxh| + |xh| mean |dxh xh|) with |dxh| bounded by 1.2 |dy w| (the tanh
  GELU's slope stays below 1.13): the size of the terms that meet in dx.
  bf16 adds one bf16 ulp of the result (the final rounding).
- dw, db: sums over M rows, added in fixed order (the rows of one CTA, then
  the CTA partials, at most 4096, in 32 strided sums and a sum of those): within
  (u (ceil(M / min(M, 152)) + 512) + 2e-6) A with A = 1.2 sum over the rows of
  |dy xh| (dw) or |dy| (db); 512 bounds the additions after the CTA level.
  dw adds 8 u 1.2 sum |dy|: xh = (x - mean) rstd from fp32 statistics is off
  by a few u in absolute terms (the mean's residual), which a row whose xh is
  near 0 shows in relative terms (visible with a single row).
At full size a sparse dy (zero except on sampled rows) pins every row's
contribution: dx must be exactly 0 on the other rows and dw, db must be the
sums over the sampled rows alone.
"""
import math

import numpy as np
import pytest
import torch

from row_wise_reduction_gb300 import (rowops_device_status, rowops_layernorm_gelu_backward,
                                      rowops_layernorm_gelu_backward_workspace_bytes, workloads)
from tests import _compare as C
from tests import gpu_util as gu

pytestmark = [pytest.mark.gpu, gu.requires_gpu]

B1 = workloads.WORKLOADS["layernorm_gelu_backward_f32_4096x768"]
B2 = workloads.WORKLOADS["layernorm_gelu_backward_bf16_65536x8192"]
U = 2.0 ** -24


def edge(dtype, M, N, seed=21, x_std=1.0):
    return workloads.Workload(f"edge_bwd_{dtype}_{M}x{N}", "layernorm_gelu_backward", dtype, M, N, seed=seed,
                              x_std=x_std, affine=True, grad=True)


def host(t):
    return None if t is None else t.float().cpu().numpy()


def scales(x, dy, w, eps):
    """S (dx elementwise) and A_w, A_b (dw, db per column) in float64."""
    x = x.astype(np.float64)
    dy = dy.astype(np.float64)
    wa = np.ones(x.shape[1]) if w is None else np.abs(w.astype(np.float64))
    mean = x.mean(axis=1, keepdims=True)
    rstd = 1.0 / np.sqrt(((x - mean) ** 2).mean(axis=1, keepdims=True) + eps)
    xh = (x - mean) * rstd
    dxh = 1.2 * np.abs(dy) * wa
    S = rstd * (dxh + dxh.mean(axis=1, keepdims=True) + np.abs(xh) * (dxh * np.abs(xh)).mean(axis=1, keepdims=True))
    return S, 1.2 * np.abs(dy * xh).sum(axis=0), 1.2 * np.abs(dy).sum(axis=0)


def assert_dx_close(got, ref, S, dtype, what):
    tol = 1e-5 * S
    if dtype == "bf16":
        tol = tol + C.bf16_ulp(ref)
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    assert not bad.any(), (f"{what}: dx off at {np.argwhere(bad)[:5].tolist()}: got {got[bad][:5]}, "
                           f"want {ref[bad][:5]}, tol {tol[bad][:5]}")


def assert_sum_close(got, ref, A, M, what, A_dy=None):
    n_add = math.ceil(M / min(M, 152)) + 512
    tol = (U * n_add + 2e-6) * A
    if A_dy is not None:  # dw: xh carries an absolute error of a few u (fp32 statistics), times |dz| per row
        tol = tol + 8 * U * A_dy
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    assert not bad.any(), (f"{what}: off at columns {np.argwhere(bad)[:5].ravel().tolist()}: got {got[bad][:5]}, "
                           f"want {ref[bad][:5]}, tol {tol[bad][:5]}")


def run(x, dy, w, b, eps, dx=None):
    dx, dw, db = rowops_layernorm_gelu_backward(x, dy, w, b, eps, dx=dx)
    torch.cuda.synchronize()
    assert rowops_device_status() == 0
    return dx, dw, db


def check(oracle, wl, ld=None, offset=0, dy_offset=0, dx_offset=None, use_affine=True):
    inp = gu.make_x(wl, ld=ld, offset=offset)
    x = inp["x"]
    ldx = x.stride(0) if wl.M > 1 else wl.N
    dy = inp["dy"] if not dy_offset else place(inp["dy"], ldx, dy_offset)
    w = inp.get("w") if use_affine else None
    b = inp.get("b") if use_affine else None
    dx, buf, inside = gu.guarded_like(x, offset=offset if dx_offset is None else dx_offset)
    run(x, dy, w, b, wl.eps, dx=dx)
    xin, gin = gu.rows_f32(x), gu.rows_f32(dy)
    ref_dx, ref_dw, ref_db = oracle.layernorm_gelu_backward(xin, gin, host(w), host(b), wl.eps)
    S, Aw, Ab = scales(xin, gin, host(w), wl.eps)
    assert_dx_close(C.to_f64(dx), ref_dx, S, wl.dtype, wl.name)
    gu.assert_guard_untouched(buf, inside)
    return x, dy, w, b, (ref_dw, Aw), (ref_db, Ab)


def place(t: torch.Tensor, ld: int, offset: int):
    M, N = t.shape
    buf = torch.full((M * ld + offset + 8,), float("nan"), dtype=t.dtype, device=t.device)
    view = torch.as_strided(buf, (M, N), (ld, 1), offset)
    view.copy_(t)
    return view


def check_all(oracle, wl, **kw):
    x, dy, w, b, (rw, Aw), (rb, Ab) = check(oracle, wl, **kw)
    _, dw, db = run(x, dy, w, b, wl.eps)
    assert_sum_close(C.to_f64(dw), rw, Aw, wl.M, wl.name + " dw", A_dy=Ab)
    assert_sum_close(C.to_f64(db), rb, Ab, wl.M, wl.name + " db")


def test_f32_workload_in_full(oracle):
    check_all(oracle, B1)


def test_bf16_workload_reduced_rows(oracle):
    check_all(oracle, B2.with_shape(M=512))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [256, 512, 768, 1024, 1536, 2048, 3072, 4096, 6144, 8192, 12288, 16384])
def test_widths(oracle, dtype, N):
    """Widths up to 16384: those with a row-pipeline tile (TPR x VPT vectors of
    at most 16 columns per thread) and the rest on the looped kernel."""
    check_all(oracle, edge(dtype, 700, N))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 2, 7, 127, 255, 1000, 4097, 20000, 40000])
def test_looped_widths(oracle, dtype, N):
    """Widths without a tile (ragged, tiny, longer than the ring): the looped kernel."""
    check_all(oracle, edge(dtype, 300, N))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_strided_and_misaligned_rows(oracle, dtype):
    es = workloads.elem_size(dtype)
    for ld, off, dyo, dxo in [(1040, 0, 0, 0), (1029, 0, 0, 0), (1024, 1, 0, 1), (1024, 0, 3, 5),
                              (1032, 4 // es if es < 4 else 1, 0, 0)]:
        check_all(oracle, edge(dtype, 200, 1024), ld=ld, offset=off, dy_offset=dyo, dx_offset=dxo)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_no_affine(oracle, dtype):
    check_all(oracle, edge(dtype, 256, 2048), use_affine=False)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_few_rows(oracle, dtype):
    for M in (1, 2, 3, 151, 153):
        check_all(oracle, edge(dtype, M, 1024))


def test_shifted_and_scaled_rows(oracle):
    """Rows far from zero and rows of tiny spread: the statistics are those of
    the forward (centred, corrected), so xh stays accurate."""
    wl = edge("f32", 256, 1024, x_std=1e-3)
    inp = gu.make_x(wl)
    x = inp["x"]
    x.add_(100.0)
    dy, w, b = inp["dy"], inp["w"], inp["b"]
    dx, dw, db = run(x, dy, w, b, wl.eps)
    xin, gin = gu.rows_f32(x), gu.rows_f32(dy)
    ref_dx, ref_dw, ref_db = oracle.layernorm_gelu_backward(xin, gin, host(w), host(b), wl.eps)
    S, Aw, Ab = scales(xin, gin, host(w), wl.eps)
    assert_dx_close(C.to_f64(dx), ref_dx, S, "f32", "shifted rows")
    assert_sum_close(C.to_f64(db), ref_db, Ab, wl.M, "db")


def test_constant_rows(oracle):
    """x constant along a row: xh = 0, rstd = 1 / sqrt(eps); dx = rstd (dxh - mean dxh)."""
    wl = edge("f32", 64, 1024)
    inp = gu.make_x(wl)
    x = inp["x"]
    x.copy_(torch.linspace(-3, 3, 64, device=x.device).unsqueeze(1).expand(64, 1024))
    dy, w, b = inp["dy"], inp["w"], inp["b"]
    dx, dw, db = run(x, dy, w, b, wl.eps)
    xin, gin = gu.rows_f32(x), gu.rows_f32(dy)
    ref_dx, ref_dw, ref_db = oracle.layernorm_gelu_backward(xin, gin, host(w), host(b), wl.eps)
    S, Aw, Ab = scales(xin, gin, host(w), wl.eps)
    assert_dx_close(C.to_f64(dx), ref_dx, S, "f32", "constant rows")
    # xh = 0 in exact arithmetic; fp32 leaves at most rounding residue of the mean
    assert np.all(np.abs(C.to_f64(dw)) <= 1e-6 * Ab)
    assert_sum_close(C.to_f64(db), ref_db, Ab, wl.M, "db")


@pytest.mark.parametrize("dtype,N", [("bf16", 8192), ("f32", 8192), ("f32", 1024), ("bf16", 4097)])
def test_outlier_rows(oracle, dtype, N):
    """One large negative entry per row: xh reaches about -sqrt(N) there and z
    far below -10, where the tanh GELU's slope underflows to 0 (it must not
    overflow into NaN)."""
    wl = edge(dtype, 160, N)
    inp = gu.make_x(wl)
    x = inp["x"]
    cols = torch.randint(0, N, (160,), generator=torch.Generator().manual_seed(3)).to(x.device)
    x[torch.arange(160, device=x.device), cols] = -1000.0
    dy, w, b = inp["dy"], inp["w"], inp["b"]
    dx, dw, db = run(x, dy, w, b, wl.eps)
    xin, gin = gu.rows_f32(x), gu.rows_f32(dy)
    ref_dx, ref_dw, ref_db = oracle.layernorm_gelu_backward(xin, gin, host(w), host(b), wl.eps)
    S, Aw, Ab = scales(xin, gin, host(w), wl.eps)
    assert_dx_close(C.to_f64(dx), ref_dx, S, dtype, "outlier rows")
    assert_sum_close(C.to_f64(dw), ref_dw, Aw, wl.M, "dw", A_dy=Ab)
    assert_sum_close(C.to_f64(db), ref_db, Ab, wl.M, "db")


@pytest.mark.parametrize("ring", ["2", "3", "4", "5", "6"])
@pytest.mark.parametrize("dtype,N", [("bf16", 8192), ("bf16", 2048), ("f32", 3072)])
def test_ring_depths(oracle, monkeypatch, ring, dtype, N):
    """Partials in registers: ROWOPS_RING_BUFFERS below 4 selects the
    one-row-at-a-time kernel, 4 and up the three-stage pipeline: both against
    the oracle, with few rows per CTA and with many."""
    monkeypatch.setenv("ROWOPS_BWD_PARTIALS", "registers")
    monkeypatch.setenv("ROWOPS_RING_BUFFERS", ring)
    for M in (157, 2000):
        check_all(oracle, edge(dtype, M, N, seed=int(ring) + M))


@pytest.mark.parametrize("ring", ["2", "3", "4"])
@pytest.mark.parametrize("dtype,N", [("bf16", 8192), ("bf16", 4096), ("bf16", 2048), ("bf16", 1024), ("f32", 4096),
                                     ("f32", 2048), ("f32", 1024), ("f32", 512)])
def test_tmem_partials(oracle, monkeypatch, ring, dtype, N):
    """Partials in tensor memory (the default where a 512-thread CTA of two row
    groups of 256 threads, or four of 128, covers the row with at most 32
    columns a thread): against the oracle with fewer rows than row groups, a
    few rows per group and many; ring depths 3 and 4 where they fit."""
    monkeypatch.setenv("ROWOPS_BWD_PARTIALS", "tmem")
    monkeypatch.setenv("ROWOPS_RING_BUFFERS", ring)
    for M in (1, 3, 157, 2000):
        check_all(oracle, edge(dtype, M, N, seed=int(ring) * 31 + M))


def test_tmem_and_register_partials_agree():
    """The two forms of the dw, db partials on the same inputs: dx within a
    bf16 ulp of each other (the statistics are formed in another order), dw
    and db sums of nearly the same terms in another order (close)."""
    import os
    from row_wise_reduction_gb300 import rowops_reload_tuning
    wl = edge("bf16", 3000, 8192, seed=77)
    inp = gu.make_x(wl)
    out = {}
    for form in ("tmem", "registers"):
        os.environ["ROWOPS_BWD_PARTIALS"] = form
        rowops_reload_tuning()
        try:
            out[form] = run(inp["x"], inp["dy"], inp["w"], inp["b"], wl.eps)
        finally:
            del os.environ["ROWOPS_BWD_PARTIALS"]
            rowops_reload_tuning()
    (dx1, dw1, db1), (dx2, dw2, db2) = out["tmem"], out["registers"]
    a, c = C.to_f64(dx1), C.to_f64(dx2)
    assert np.all(np.abs(a - c) <= C.bf16_ulp(c) + 1e-6)
    torch.testing.assert_close(dw1, dw2, rtol=1e-5, atol=1e-3)
    torch.testing.assert_close(db1, db2, rtol=1e-5, atol=1e-3)


@pytest.mark.parametrize("dtype,N,vpt", [("bf16", 8192, "1"), ("bf16", 8192, "2"), ("f32", 4096, "1"),
                                         ("f32", 4096, "2"), ("bf16", 4096, "1")])
def test_row_group_widths(oracle, monkeypatch, dtype, N, vpt):
    """ROWOPS_FORCE_VPT picks the tile: 1024 threads of 8 columns or 512 of 16
    (bf16 8192), and so on."""
    monkeypatch.setenv("ROWOPS_FORCE_VPT", vpt)
    for M in (100, 1500):
        check_all(oracle, edge(dtype, M, N, seed=int(vpt) * 7 + M))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_rows(dtype):
    wl = edge(dtype, 4, 256)
    inp = gu.make_x(wl)
    x = inp["x"][:0]
    dw = torch.full((256,), 7.0, device=x.device)
    db = torch.full((256,), 7.0, device=x.device)
    dx, dw, db = rowops_layernorm_gelu_backward(x, inp["dy"][:0], inp["w"], inp["b"], 1e-5, dw=dw, db=db)
    torch.cuda.synchronize()
    assert dx.shape == (0, 256)
    assert torch.all(dw == 0) and torch.all(db == 0)


@pytest.mark.parametrize("N", [8192, 4097])
def test_deterministic(N):
    """Two calls give the same bits (fixed reduction order)."""
    wl = edge("bf16", 20000, N)
    inp = gu.make_x(wl)
    r1 = rowops_layernorm_gelu_backward(inp["x"], inp["dy"], inp["w"], inp["b"], 1e-5)
    r2 = rowops_layernorm_gelu_backward(inp["x"], inp["dy"], inp["w"], inp["b"], 1e-5)
    torch.cuda.synchronize()
    for a, c in zip(r1, r2):
        assert torch.equal(a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32),
                           c.view(torch.int16 if c.dtype == torch.bfloat16 else torch.int32))


def test_workspace_reuse_and_size():
    wl = edge("f32", 1000, 1024)
    inp = gu.make_x(wl)
    need = rowops_layernorm_gelu_backward_workspace_bytes(1000, 1024, torch.float32)
    ws = torch.empty(need, dtype=torch.uint8, device=inp["x"].device)
    a = rowops_layernorm_gelu_backward(inp["x"], inp["dy"], inp["w"], inp["b"], 1e-5, workspace=ws)
    b = rowops_layernorm_gelu_backward(inp["x"], inp["dy"], inp["w"], inp["b"], 1e-5, workspace=ws)
    torch.cuda.synchronize()
    assert all(torch.equal(p, q) for p, q in zip(a, b))
    from row_wise_reduction_gb300 import RowopsError
    with pytest.raises(RowopsError):
        rowops_layernorm_gelu_backward(inp["x"], inp["dy"], inp["w"], inp["b"], 1e-5, workspace=ws[: need - 256])


def test_full_size_sparse_dy(oracle):
    """The bf16 65536 x 8192 workload with dy zero except on 48 sampled rows
    (first, last and across the CTAs): dx exactly 0 elsewhere, the sampled rows'
    dx and the column sums against the oracle run on those rows alone."""
    inp = gu.make_x(B2)
    x, dyfull, w, b = inp["x"], inp["dy"], inp["w"], inp["b"]
    rows = np.unique(np.concatenate([gu.sample_rows(B2.M, 46, seed=5), [0, B2.M - 1]]))
    dy = torch.zeros_like(dyfull)
    idx = torch.as_tensor(rows, device=x.device)
    dy[idx] = dyfull[idx]
    del dyfull
    dx, dw, db = run(x, dy, w, b, B2.eps)
    keep = torch.zeros(B2.M, dtype=torch.bool, device=x.device)
    keep[idx] = True
    assert torch.all(dx[~keep] == 0), "rows with dy = 0 must get dx = 0"
    xin, gin = gu.rows_f32(x, rows), gu.rows_f32(dy, rows)
    ref_dx, ref_dw, ref_db = oracle.layernorm_gelu_backward(xin, gin, host(w), host(b), B2.eps)
    S, Aw, Ab = scales(xin, gin, host(w), B2.eps)
    assert_dx_close(C.to_f64(dx[idx]), ref_dx, S, "bf16", "sampled rows")
    assert_sum_close(C.to_f64(dw), ref_dw, Aw, len(rows) + 152, "dw", A_dy=Ab)
    assert_sum_close(C.to_f64(db), ref_db, Ab, len(rows) + 152, "db")


def test_full_size_dense(oracle):
    """The bf16 65536 x 8192 workload as the bench runs it: dx on sampled rows
    against the oracle; dw, db within the bound of their two-level sums, from
    the oracle's full double sums."""
    inp = gu.make_x(B2)
    x, dy, w, b = inp["x"], inp["dy"], inp["w"], inp["b"]
    dx, dw, db = run(x, dy, w, b, B2.eps)
    rows = gu.sample_rows(B2.M, 32, seed=9)
    xin, gin = gu.rows_f32(x, rows), gu.rows_f32(dy, rows)
    ref_dx, _, _ = oracle.layernorm_gelu_backward(xin, gin, host(w), host(b), B2.eps)
    S, _, _ = scales(xin, gin, host(w), B2.eps)
    assert_dx_close(C.to_f64(dx[torch.as_tensor(rows, device=x.device)]), ref_dx, S, "bf16", "sampled rows")
    # column sums over all rows, 4096 rows at a time
    ref_dw = np.zeros(B2.N)
    ref_db = np.zeros(B2.N)
    Aw = np.zeros(B2.N)
    Ab = np.zeros(B2.N)
    for r0 in range(0, B2.M, 4096):
        xs, gs = gu.rows_f32(x[r0:r0 + 4096]), gu.rows_f32(dy[r0:r0 + 4096])
        _, pw, pb = oracle.layernorm_gelu_backward(xs, gs, host(w), host(b), B2.eps)
        _, aw, ab = scales(xs, gs, host(w), B2.eps)
        ref_dw += pw
        ref_db += pb
        Aw += aw
        Ab += ab
    assert_sum_close(C.to_f64(dw), ref_dw, Aw, B2.M, "dw", A_dy=Ab)
    assert_sum_close(C.to_f64(db), ref_db, Ab, B2.M, "db")
