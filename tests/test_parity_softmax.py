"""GPU parity of rowops_softmax with the oracle, called through the C ABI.

Full-tensor comparisons at sizes the oracle finishes in seconds (several row
groups and ragged tails), the full 32768 x 4096 bf16 causal workload in the
benchmark's launch configuration on sampled rows plus size-independent
properties, and edge cases: tiny / ragged / huge N, strided and misaligned
rows, in place, masked / NaN rows, every kernel variant, guard bands.
"""
import numpy as np
import pytest
import torch

from row_wise_reduction_gb300 import rowops_softmax, workloads
from tests import _compare as C
from tests import gpu_util as gu

pytestmark = [pytest.mark.gpu, gu.requires_gpu]

W1 = workloads.WORKLOADS["softmax_f32_1024x768"]
W3 = workloads.WORKLOADS["softmax_bf16_causal_32768x4096"]


def edge(dtype, M, N, seed=7, std=3.0):
    return workloads.Workload(f"edge_{dtype}_{M}x{N}", "softmax", dtype, M, N, seed=seed, x_std=std)


def check(oracle, wl, ld=None, offset=0, yoffset=None, inplace=False):
    inp = gu.make_x(wl, ld=ld, offset=offset)
    x = inp["x"]
    xin = gu.rows_f32(x)
    if inplace:
        y = x
        buf = inside = None
    else:
        y, buf, inside = gu.guarded_like(x, offset=offset if yoffset is None else yoffset)
    rowops_softmax(x, y)
    torch.cuda.synchronize()
    ref = oracle.softmax(xin)
    err = C.assert_softmax_close(C.to_f64(y), ref, wl.dtype, what=wl.name)
    if buf is not None:
        gu.assert_guard_untouched(buf, inside)
    return err


def test_softmax_f32_1024x768_full(oracle):
    check(oracle, W1)


@pytest.mark.parametrize("M", [1024, 4096 + 37])
def test_softmax_bf16_causal_reduced_rows(oracle, M):
    """The causal bf16 workload on its first M rows (every row length of the
    mask pattern from 1 to min(M, 4096) kept entries)."""
    check(oracle, W3.with_shape(M=M))


def test_softmax_bf16_causal_full_size_sampled(oracle):
    """Full 32768 x 4096 bf16 causal workload, default launch configuration:
    64 sampled rows against the oracle; on every row, masked entries are
    exactly 0 and the row sums to 1 within bf16 rounding."""
    inp = gu.make_x(W3)
    x = inp["x"]
    y = rowops_softmax(x)
    torch.cuda.synchronize()
    rows = gu.sample_rows(W3.M, 64, seed=3)
    ref = oracle.softmax(gu.rows_f32(x, rows))
    C.assert_softmax_close(C.to_f64(y[torch.as_tensor(rows, device=y.device)]), ref, "bf16")
    masked = torch.isneginf(x)
    assert torch.all(y[masked] == 0)
    sums = y.float().sum(dim=1)
    assert torch.all((sums - 1).abs() <= 2.0 ** -8)
    del x, y, inp


RAGGED_N = [1, 2, 3, 7, 8, 9, 15, 16, 17, 31, 33, 127, 128, 129, 255, 767, 768, 769, 1000, 4095, 4096,
            4097, 8191, 16384, 16385, 32768, 32769, 100003]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", RAGGED_N)
def test_softmax_ragged_n(oracle, dtype, N):
    """Every row length class: sub-vector rows, ragged tails, the largest
    register-resident rows (16384 fp32 / 32768 bf16) and looped rows beyond."""
    check(oracle, edge(dtype, 37, N))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,ld,offset", [(127, 127, 0), (127, 127, 1), (4097, 4097, 3), (768, 773, 0),
                                         (768, 832, 5), (100003, 100010, 1), (5, 13, 2)])
def test_softmax_strided_and_misaligned_rows(oracle, dtype, N, ld, offset):
    """ld > N with NaN padding (never read), rows whose starts are not 16-byte
    aligned (peeled head / tail), in both kernel families."""
    check(oracle, edge(dtype, 29, N, seed=N + ld), ld=ld, offset=offset)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [127, 4097, 20000])
def test_softmax_x_and_y_out_of_phase(oracle, dtype, N):
    """x and y rows at different offsets modulo 16 bytes: the element-wise path."""
    check(oracle, edge(dtype, 9, N), offset=1, yoffset=0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [768, 4096, 50000])
def test_softmax_in_place(oracle, dtype, N):
    check(oracle, edge(dtype, 17, N), inplace=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [300, 40000])
def test_softmax_special_rows(oracle, dtype, N):
    """All-masked row -> zeros; NaN row -> NaN; one unmasked entry -> 1; a
    +30 outlier; a row far below zero; a row of equal values -> 1/N."""
    g = torch.Generator().manual_seed(N)
    x = torch.randn(8, N, generator=g) * 2
    x[0] = float("-inf")
    x[1, N // 3] = float("nan")
    x[2] = float("-inf")
    x[2, N - 1] = 4.0
    x[3, 5] = 30.0
    x[4] -= 1e4
    x[5] = 0.25
    x[6, ::2] = float("-inf")
    xt = x.to(workloads.torch_dtype(dtype)).cuda()
    y = rowops_softmax(xt)
    torch.cuda.synchronize()
    ref = oracle.softmax(xt.float().cpu().numpy())
    C.assert_softmax_close(C.to_f64(y), ref, dtype)
    yy = y.float().cpu()
    assert torch.all(yy[0] == 0)
    assert torch.all(torch.isnan(yy[1]))
    assert yy[2, N - 1] == 1.0 and torch.all(yy[2, : N - 1] == 0)


def test_softmax_deterministic():
    wl = edge("bf16", 513, 4096)
    x = gu.make_x(wl)["x"]
    a = rowops_softmax(x)
    b = rowops_softmax(x)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_softmax_empty_is_noop():
    x = torch.empty(0, 64, device="cuda")
    y = rowops_softmax(x)
    torch.cuda.synchronize()
    assert y.shape == (0, 64)


VARIANTS = [(tpr, vpt) for tpr in (16, 32, 64, 128, 256, 512, 1024) for vpt in (1, 2, 3, 4)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("tpr,vpt", VARIANTS)
def test_softmax_every_register_variant(oracle, monkeypatch, dtype, tpr, vpt):
    """Each register-resident instantiation, forced, on the largest row it
    holds minus a ragged tail, on a misaligned base."""
    vec = 4 if dtype == "f32" else 8
    N = tpr * vpt * vec - 3
    monkeypatch.setenv("ROWOPS_KERNEL", "reg")
    monkeypatch.setenv("ROWOPS_FORCE_TPR", str(tpr))
    monkeypatch.setenv("ROWOPS_FORCE_VPT", str(vpt))
    check(oracle, edge(dtype, 2 * (1024 // tpr) + 3, N, seed=tpr * 10 + vpt), offset=1)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("ctas", ["-1", "1", "2"])
def test_softmax_grid_modes(oracle, monkeypatch, dtype, ctas):
    """Persistent grids of 1 and 2 CTAs per SM and the one-CTA-per-row-group
    grid give the oracle's result (rows handed out by the grid-stride loop)."""
    monkeypatch.setenv("ROWOPS_CTAS_PER_SM", ctas)
    check(oracle, edge(dtype, 3001, 768))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_softmax_forced_looped(oracle, monkeypatch, dtype):
    monkeypatch.setenv("ROWOPS_FORCE_LOOPED", "1")
    check(oracle, edge(dtype, 65, 4097), offset=2)


TMA_VARIANTS = [(b, v) for b in (64, 128, 256, 512) for v in (1, 2, 3, 4, 8)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("block,vpt", TMA_VARIANTS)
@pytest.mark.parametrize("full", [True, False])
def test_softmax_every_tma_variant(oracle, monkeypatch, dtype, block, vpt, full):
    """Each TMA-fed row-pipeline instantiation, forced: rows of exactly
    block * vpt vectors (no predicates) and rows one vector shorter."""
    vec = 4 if dtype == "f32" else 8
    nvec = block * vpt - (0 if full else 1)
    if nvec < 64:
        pytest.skip("the row pipeline takes rows of at least 64 vectors")
    monkeypatch.setenv("ROWOPS_KERNEL", "tma")
    monkeypatch.setenv("ROWOPS_FORCE_TPR", str(block))
    monkeypatch.setenv("ROWOPS_FORCE_VPT", str(vpt))
    check(oracle, edge(dtype, 3 * 152 + 5, nvec * vec, seed=block + vpt))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("ring", ["2", "3", "7", "16"])
@pytest.mark.parametrize("ctas", ["0", "1", "-1"])
def test_softmax_tma_ring_depths_and_grids(oracle, monkeypatch, dtype, ring, ctas):
    """Ring depths (rows in flight per CTA) with persistent and one-row-per-CTA
    grids; 1000 rows so every CTA wraps around its ring several times."""
    monkeypatch.setenv("ROWOPS_KERNEL", "tma")
    monkeypatch.setenv("ROWOPS_RING_BUFFERS", ring)
    monkeypatch.setenv("ROWOPS_CTAS_PER_SM", ctas)
    check(oracle, edge(dtype, 1000, 2048))
    from row_wise_reduction_gb300 import rowops_device_status

    assert rowops_device_status() == 0


def test_softmax_tma_in_place_and_strided(oracle, monkeypatch):
    monkeypatch.setenv("ROWOPS_KERNEL", "tma")
    check(oracle, edge("bf16", 301, 4096), inplace=True)
    check(oracle, edge("bf16", 301, 4096), ld=4096 + 64)
    check(oracle, edge("f32", 77, 1024), ld=1024 + 4)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N,ld,offset", [(4097, 4097, 0), (8191, 8191, 0), (1000, 1003, 1), (3001, 3001, 2),
                                         (12345, 12350, 1)])
def test_softmax_tma_general_rows(oracle, monkeypatch, dtype, N, ld, offset):
    """The row pipeline's general form on rows that start anywhere."""
    monkeypatch.setenv("ROWOPS_KERNEL", "tma")
    check(oracle, edge(dtype, 157, N, seed=N + ld), ld=ld, offset=offset)
    from row_wise_reduction_gb300 import rowops_device_status

    assert rowops_device_status() == 0
