"""The library's calls captured in a CUDA graph: each captured once (after one
ordinary call), then replayed on new inputs written into the captured
buffers; every replay is checked against the oracle on sampled rows. The
calls take the current stream, so inside `torch.cuda.graph` they are recorded
into the graph: kernels, the cooperative launch of the row-group form (which
zeroes its own slots), the programmatic dependent launch of the two-launch
form, and the backward's tensor-memory kernel with its fixed-order reduce."""
import pytest
import torch

from row_wise_reduction_gb300 import (
    rowops_layernorm_gelu,
    rowops_layernorm_gelu_backward,
    rowops_layernorm_gelu_backward_workspace_bytes,
    rowops_online_softmax,
    rowops_online_softmax_status,
    rowops_online_softmax_workspace_bytes,
    rowops_softmax,
)
from tests import _compare as C
from tests import gpu_util as gu

pytestmark = [pytest.mark.gpu, gu.requires_gpu]


def _fill(t, seed, std=3.0):
    g = torch.Generator(device=t.device).manual_seed(seed)
    t.copy_(torch.randn(t.shape, device=t.device, generator=g) * std)


@pytest.mark.parametrize("M,N", [(40, 1 << 18), (8, 1 << 17)])
def test_online_softmax_replayed_from_a_cuda_graph(oracle, M, N):
    """40 x 2^18 fp32 takes the single-kernel row-group form (one cooperative
    kernel); 8 x 2^17 the two-launch form (the second launch a programmatic
    dependent of the first)."""
    x = torch.empty(M, N, device="cuda")
    y = torch.empty_like(x)
    ws = torch.empty(rowops_online_softmax_workspace_bytes(M, N, x.dtype), dtype=torch.uint8, device="cuda")
    _fill(x, 100)
    rowops_online_softmax(x, y, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rowops_online_softmax(x, y, workspace=ws)
    for seed in range(3):
        _fill(x, seed)
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert rowops_online_softmax_status(ws) == 0
        rows = gu.sample_rows(M, 3, seed=seed)
        ref = oracle.softmax(gu.rows_f32(x, rows))
        C.assert_softmax_close(C.to_f64(y[torch.as_tensor(rows, device=y.device)]), ref, "f32",
                               what=f"graph replay {seed}")


def test_softmax_and_layernorm_gelu_replayed_from_one_cuda_graph(oracle):
    """A bf16 softmax and a bf16 LayerNorm+GELU captured into one graph."""
    xs = torch.empty(256, 4096, device="cuda", dtype=torch.bfloat16)
    ys = torch.empty_like(xs)
    xl = torch.empty(512, 8192, device="cuda", dtype=torch.bfloat16)
    yl = torch.empty_like(xl)
    w = torch.empty(8192, device="cuda", dtype=torch.bfloat16)
    b = torch.empty_like(w)
    _fill(w, 7, 1.0)
    _fill(b, 8, 1.0)
    eps = 1e-5
    _fill(xs, 200)
    _fill(xl, 201)
    rowops_softmax(xs, ys)
    rowops_layernorm_gelu(xl, w, b, eps, yl)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rowops_softmax(xs, ys)
        rowops_layernorm_gelu(xl, w, b, eps, yl)
    wn, bn = w.float().cpu().numpy(), b.float().cpu().numpy()
    for seed in range(3):
        _fill(xs, 10 + seed)
        _fill(xl, 20 + seed)
        g.replay()
        torch.cuda.synchronize()
        rs = gu.sample_rows(256, 4, seed=seed)
        C.assert_softmax_close(C.to_f64(ys[torch.as_tensor(rs, device=ys.device)]),
                               oracle.softmax(gu.rows_f32(xs, rs)), "bf16", what=f"softmax replay {seed}")
        rl = gu.sample_rows(512, 4, seed=seed)
        C.assert_ln_gelu_close(C.to_f64(yl[torch.as_tensor(rl, device=yl.device)]),
                               oracle.layernorm_gelu(gu.rows_f32(xl, rl), wn, bn, eps), "bf16")


def test_layernorm_gelu_backward_replayed_from_a_cuda_graph(oracle):
    """bf16 600 x 8192: the tensor-memory kernel (each CTA allocates and frees
    its TMEM columns in every replay) and the reduce kernel of dw, db, against
    the oracle at the backward's tolerances."""

    M, N, eps = 600, 8192, 1e-5
    x = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    dy = torch.empty_like(x)
    dx = torch.empty_like(x)
    w = torch.empty(N, device="cuda", dtype=torch.bfloat16)
    b = torch.empty_like(w)
    dw = torch.empty(N, device="cuda")
    db = torch.empty_like(dw)
    ws = torch.empty(rowops_layernorm_gelu_backward_workspace_bytes(M, N, x.dtype), dtype=torch.uint8, device="cuda")
    _fill(w, 30, 0.5)
    _fill(b, 31, 0.1)
    _fill(x, 32, 1.0)
    _fill(dy, 33, 1.0)
    rowops_layernorm_gelu_backward(x, dy, w, b, eps, dx, dw, db, ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rowops_layernorm_gelu_backward(x, dy, w, b, eps, dx, dw, db, ws)
    from tests.test_parity_ln_gelu_backward import assert_dx_close, assert_sum_close, scales

    wn, bn = w.float().cpu().numpy(), b.float().cpu().numpy()
    for seed in range(2):
        _fill(x, 40 + seed, 1.0)
        _fill(dy, 50 + seed, 1.0)
        dx.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        xin, gin = gu.rows_f32(x), gu.rows_f32(dy)
        ref_dx, ref_dw, ref_db = oracle.layernorm_gelu_backward(xin, gin, wn, bn, eps)
        S, Aw, Ab = scales(xin, gin, wn, eps)
        assert_dx_close(C.to_f64(dx), ref_dx, S, "bf16", f"graph replay {seed}")
        assert_sum_close(C.to_f64(dw), ref_dw, Aw, M, "dw", A_dy=Ab)
        assert_sum_close(C.to_f64(db), ref_db, Ab, M, "db")
