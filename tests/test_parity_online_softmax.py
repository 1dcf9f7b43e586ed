"""GPU parity of rowops_online_softmax (split-row (m, d) partials merged in a
second pass) with the oracle and with rowops_softmax, through the C ABI."""
import math

import numpy as np
import pytest
import torch

from row_wise_reduction_gb300 import (
    rowops_online_softmax,
    rowops_online_softmax_status,
    rowops_online_softmax_workspace_bytes,
    rowops_softmax,
    workloads,
)
from tests import _compare as C
from tests import gpu_util as gu

pytestmark = [pytest.mark.gpu, gu.requires_gpu]

W4 = workloads.WORKLOADS["online_softmax_f32_64x1048576"]


def edge(dtype, M, N, seed=13, std=3.0, outlier_p=0.0):
    return workloads.Workload(f"edge_{dtype}_{M}x{N}", "online_softmax", dtype, M, N, seed=seed, x_std=std,
                              outlier_p=outlier_p)


def workspace(x):
    n = rowops_online_softmax_workspace_bytes(x.shape[0], x.shape[1], x.dtype)
    return torch.empty(n, dtype=torch.uint8, device=x.device)


def check(oracle, wl, chunk=0, ld=None, offset=0, yoffset=None, inplace=False):
    inp = gu.make_x(wl, ld=ld, offset=offset)
    x = inp["x"]
    xin = gu.rows_f32(x)
    ws = workspace(x)
    if inplace:
        y, buf, inside = x, None, None
    else:
        y, buf, inside = gu.guarded_like(x, offset=offset if yoffset is None else yoffset)
    rowops_online_softmax(x, y, workspace=ws, chunk=chunk)
    assert rowops_online_softmax_status(ws) == 0
    ref = oracle.softmax(xin)
    C.assert_softmax_close(C.to_f64(y), ref, wl.dtype, what=f"{wl.name} chunk={chunk}")
    if buf is not None:
        gu.assert_guard_untouched(buf, inside)
    return y


@pytest.mark.parametrize("chunk", [0, 4096, 65536])
def test_online_softmax_reduced_rows(oracle, chunk):
    """The 2^20-column outlier workload on its first 4 rows, at the automatic
    chunk size and at two explicit ones (256 and 16 chunks per row)."""
    check(oracle, W4.with_shape(M=4), chunk=chunk)


@pytest.mark.parametrize("form", ["default", "two_pass"])
def test_online_softmax_full_size(oracle, monkeypatch, form):
    """Full 64 x 2^20 fp32 workload, in the default launch configuration (the
    single-kernel row-group form at this size) and in the two-launch form: 4
    sampled rows against the oracle; on every row the outlier entries equal
    1 / (k + S) (k outliers, S = sum of exp(x - 30) over the rest, accumulated
    here in float64) and every row sums to 1."""
    if form == "two_pass":
        monkeypatch.setenv("ROWOPS_ONLINE", "two_pass")
    inp = gu.make_x(W4)
    x = inp["x"]
    ws = workspace(x)
    y = rowops_online_softmax(x, workspace=ws)
    assert rowops_online_softmax_status(ws) == 0
    rows = gu.sample_rows(W4.M, 4, seed=1)
    ref = oracle.softmax(gu.rows_f32(x, rows))
    C.assert_softmax_close(C.to_f64(y[torch.as_tensor(rows, device=y.device)]), ref, "f32")
    hit = x == 30.0
    k = hit.sum(dim=1, dtype=torch.float64)
    S = torch.where(hit, 0.0, torch.exp(x.double() - 30.0)).sum(dim=1)
    want = 1.0 / (k + S)
    got = torch.where(hit, y.double(), 0.0).sum(dim=1) / k
    assert torch.all((got / want - 1).abs() <= 1e-5)
    assert torch.all((y.double().sum(dim=1) - 1).abs() <= 1e-4)
    del x, y, inp


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_online_softmax_row_groups_strided_many_rows(oracle, dtype):
    """Default dispatch on a batch above 32 MiB of rows of 1 MiB (fp32) or
    512 KiB (bf16) with a padded row stride: the single-kernel row-group form
    with groups of 19 CTAs and 8 rows per wave over 5 (fp32) or 10 (bf16)
    waves, every row against the oracle, the output's guard band untouched."""
    N = 1 << 18
    M = 40 if dtype == "f32" else 80
    check(oracle, edge(dtype, M, N, seed=77, outlier_p=1e-3), chunk=0, ld=N + 64)


def test_online_matches_two_pass_softmax():
    """Split-row online softmax (automatic chunking and two explicit chunk
    counts) and rowops_softmax (whose
    2^20-column rows take the in-CTA online loop) agree within the softmax
    tolerance on the same input."""
    wl = W4.with_shape(M=8)
    x = gu.make_x(wl)["x"]
    y2 = rowops_softmax(x)
    for chunk in (0, 2048, 32768):
        y1 = rowops_online_softmax(x, chunk=chunk)
        torch.cuda.synchronize()
        a, b = y1.double(), y2.double()
        assert torch.all((a - b).abs() <= 1e-5 * b.abs() + C.FTZ_FLOOR)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,chunk", [(1, 0), (100, 256), (257, 256), (4097, 256), (8192, 1024), (30000, 0),
                                     (100003, 4096), (100003, 0)])
def test_online_softmax_ragged(oracle, dtype, N, chunk):
    M = 50 if N < 10000 else 6
    check(oracle, edge(dtype, M, N, seed=N, outlier_p=1e-3 if N > 1000 else 0.0), chunk=chunk)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,ld,offset,chunk", [(4097, 4097, 0, 256), (5000, 5003, 1, 512), (20000, 20000, 3, 0)])
def test_online_softmax_misaligned(oracle, dtype, N, ld, offset, chunk):
    """Rows and chunk starts that are not 16-byte aligned."""
    check(oracle, edge(dtype, 7, N, seed=ld), chunk=chunk, ld=ld, offset=offset)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_online_softmax_out_of_phase_and_in_place(oracle, dtype):
    check(oracle, edge(dtype, 5, 9000), chunk=1024, offset=1, yoffset=0)
    check(oracle, edge(dtype, 5, 9000), chunk=1024, inplace=True)


def test_online_softmax_masked_chunks(oracle):
    """Whole chunks of -inf (partials with d = 0) are skipped in the merge; an
    all-masked row gives zeros; a NaN poisons only its row."""
    N = 8192
    g = torch.Generator().manual_seed(3)
    x = torch.randn(4, N, generator=g)
    x[0, :4096] = float("-inf")
    x[1] = float("-inf")
    x[2, 777] = float("nan")
    x[3, 1024:7000] = float("-inf")
    xt = x.cuda()
    y = rowops_online_softmax(xt, chunk=1024)
    torch.cuda.synchronize()
    ref = oracle.softmax(x.numpy())
    C.assert_softmax_close(C.to_f64(y), ref, "f32")


@pytest.mark.parametrize("family", ["auto", "looped"])
@pytest.mark.parametrize("dtype,chunk", [("f32", 1024), ("f32", 2048), ("f32", 4096), ("f32", 8192),
                                         ("bf16", 2048), ("bf16", 4096), ("bf16", 8192), ("bf16", 16384)])
def test_online_softmax_full_chunks(oracle, monkeypatch, family, dtype, chunk):
    """Chunks that are whole 256-thread tiles of aligned rows stream through a
    shared-memory ring (auto); ROWOPS_KERNEL=looped keeps the register-load
    kernels. Both against the oracle, with a chunk of NaN only, one of -inf
    only, a +inf, an all -inf row, out of place and in place."""
    if family == "looped":
        monkeypatch.setenv("ROWOPS_KERNEL", "looped")
    N = 16 * chunk
    wl = edge(dtype, 9, N, seed=chunk + len(family), outlier_p=1e-3)
    check(oracle, wl, chunk=chunk)
    check(oracle, wl, chunk=chunk, inplace=True)
    x = gu.make_x(wl)["x"]
    x[0, chunk:2 * chunk] = float("nan")
    x[1, 3 * chunk:4 * chunk] = float("-inf")
    x[2, 5] = float("inf")
    x[3] = float("-inf")
    xin = gu.rows_f32(x)
    y = rowops_online_softmax(x, chunk=chunk)
    torch.cuda.synchronize()
    C.assert_softmax_close(C.to_f64(y), oracle.softmax(xin), dtype, what=f"special chunks {family} {chunk}")


def test_online_softmax_deterministic():
    x = gu.make_x(edge("f32", 16, 300000))["x"]
    a = rowops_online_softmax(x, chunk=4096)
    b = rowops_online_softmax(x, chunk=4096)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_online_softmax_empty_is_noop():
    x = torch.empty(0, 4096, device="cuda")
    y = rowops_online_softmax(x)
    torch.cuda.synchronize()
    assert y.shape == (0, 4096)


def set_single_read(monkeypatch, staging):
    """Force a single-read form: "smem" / "l2" (column slices of every row per
    CTA, staged in shared memory / L2) or "groups" (rows over row groups)."""
    monkeypatch.setenv("ROWOPS_ONLINE", "row_groups" if staging.startswith("groups") else "single_read")
    if staging == "l2":
        monkeypatch.setenv("ROWOPS_PERSIST_L2", "1")
    if staging == "groups256":
        monkeypatch.setenv("ROWOPS_FORCE_TPR", "512")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M,N", [(1, 1 << 20), (3, 1 << 20), (2, 1 << 21), (5, 1500000), (155, 1 << 20),
                                 (64, 40000)])
@pytest.mark.parametrize("staging", ["smem", "l2", "groups", "groups256"])
def test_online_softmax_single_read_form(oracle, monkeypatch, dtype, M, N, staging):
    """The persistent single-read forms, forced. smem / l2: column slices of
    every row per CTA, warp partials, one merging owner CTA per row, a ring of
    staged rows in shared memory or L2; shapes give fewer rows than the ring,
    more rows than CTAs (owners take several rows), uneven slices, a shallow
    ring (2^21 columns), and rows too short for it (which take the two-launch
    form). groups: rows spread over row groups of CTAs; the shapes give one row
    over every SM, groups widened for few rows, uneven slices, a partial last
    wave (155 rows), and short rows over groups of 4 CTAs."""
    set_single_read(monkeypatch, staging)
    check(oracle, edge(dtype, M, N, seed=M + N, outlier_p=1e-3), chunk=0)
    check(oracle, edge(dtype, min(M, 3), N, seed=5), chunk=0, inplace=True)


@pytest.mark.parametrize("staging", ["smem", "groups", "groups256"])
def test_online_softmax_single_read_special_rows(oracle, monkeypatch, staging):
    """Masked pieces, an all-masked row and a NaN row in the single-read forms."""
    set_single_read(monkeypatch, staging)
    N = 1 << 20
    g = torch.Generator().manual_seed(9)
    x = torch.randn(5, N, generator=g)
    x[0, : N // 2] = float("-inf")
    x[1] = float("-inf")
    x[2, 12345] = float("nan")
    x[3, 1000:N - 1000] = float("-inf")
    x[4, 5000:500000] = float("-inf")
    xt = x.cuda()
    ws = workspace(xt)
    y = rowops_online_softmax(xt, workspace=ws)
    assert rowops_online_softmax_status(ws) == 0
    C.assert_softmax_close(C.to_f64(y), oracle.softmax(x.numpy()), "f32")


@pytest.mark.parametrize("staging", ["smem", "groups"])
def test_online_softmax_single_read_repeated_calls_reuse_workspace(oracle, monkeypatch, staging):
    """The slots are reset before every call: calls in a row on one
    workspace, with different shapes, all match the oracle."""
    set_single_read(monkeypatch, staging)
    wl_a = edge("f32", 6, 1 << 20, seed=1, outlier_p=1e-3)
    wl_b = edge("f32", 3, 1 << 21, seed=2)
    xa = gu.make_x(wl_a)["x"]
    xb = gu.make_x(wl_b)["x"]
    n = max(rowops_online_softmax_workspace_bytes(6, 1 << 20, torch.float32),
            rowops_online_softmax_workspace_bytes(3, 1 << 21, torch.float32))
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    for x in (xa, xb, xa, xb):
        y = rowops_online_softmax(x, workspace=ws)
        assert rowops_online_softmax_status(ws) == 0
        C.assert_softmax_close(C.to_f64(y), oracle.softmax(x.cpu().numpy()), "f32")


def test_online_softmax_row_groups_workspace_never_cleared(oracle, monkeypatch):
    """The single-kernel row-group form enqueues no fill of the workspace: it
    zeroes the slots it uses itself. One workspace, first filled with random
    bytes and then left as each call leaves it, serves calls of different
    shapes (rows over 76, 38 and 19 CTAs, so slot layouts overlap with
    different strides) and of both forms in turn (the two-launch form writes
    chunk partials over the same bytes); every output matches the oracle."""
    shapes = [(64, 1 << 20, "f32", "row_groups"), (9, 1 << 20, "f32", "two_pass"), (40, 1 << 18, "f32", "row_groups"),
              (80, 1 << 18, "bf16", "row_groups"), (5, 1 << 21, "f32", "row_groups"), (64, 1 << 20, "f32", "row_groups")]
    n = max(rowops_online_softmax_workspace_bytes(M, N, workloads.torch_dtype(dt)) for M, N, dt, _ in shapes)
    g = torch.Generator(device="cuda").manual_seed(123)
    ws = torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda", generator=g)
    for i, (M, N, dt, form) in enumerate(shapes):
        monkeypatch.setenv("ROWOPS_ONLINE", form)
        wl = edge(dt, M, N, seed=100 + i, outlier_p=1e-3)
        x = gu.make_x(wl)["x"]
        y = rowops_online_softmax(x, workspace=ws)
        assert rowops_online_softmax_status(ws) == 0
        rows = gu.sample_rows(M, min(M, 6), seed=i)
        ref = oracle.softmax(gu.rows_f32(x, rows))
        C.assert_softmax_close(C.to_f64(y[torch.as_tensor(rows, device=y.device)]), ref, dt,
                               what=f"call {i}: {form} {dt} {M}x{N}")
        assert torch.all((y.double().sum(dim=1) - 1).abs() <= (1e-3 if dt == "f32" else 1e-2))
        del x, y
