"""The bounded device-side waits end in a recorded ROWOPS_ERR_TIMEOUT, not a
hang, and the CUDA context stays usable afterwards.

No GPU fault is involved: the test hook ROWOPS_TEST_STALL_ROW makes one wait
unsatisfiable (the row pipeline's mbarrier expects 16 bytes more than the bulk
copy of that row brings; the single-read split softmax withholds one partial,
a slot nothing then sets), and ROWOPS_WAIT_LIMIT_NS shortens every wait to
20 ms. The kernel gives up, drains its own copies, records the timeout and
returns; the next call without the hook is correct and clean.
"""
import numpy as np
import pytest
import torch

from row_wise_reduction_gb300 import (
    rowops_device_status,
    rowops_layernorm_gelu,
    rowops_layernorm_gelu_backward,
    rowops_online_softmax,
    rowops_online_softmax_status,
    rowops_online_softmax_workspace_bytes,
    rowops_softmax,
    workloads,
)
from tests import _compare as C
from tests import gpu_util as gu

pytestmark = [pytest.mark.gpu, gu.requires_gpu]

TIMEOUT = 5
LIMIT_NS = "20000000"


def _softmax_wl():
    return workloads.Workload("timeout_softmax", "softmax", "bf16", 2000, 4096, seed=3, x_std=2.0)


def test_row_pipeline_wait_times_out_and_context_recovers(oracle, monkeypatch):
    x = gu.make_x(_softmax_wl())["x"]
    assert rowops_device_status() == 0
    monkeypatch.setenv("ROWOPS_KERNEL", "tma")
    monkeypatch.setenv("ROWOPS_WAIT_LIMIT_NS", LIMIT_NS)
    monkeypatch.setenv("ROWOPS_TEST_STALL_ROW", "777")
    rowops_softmax(x)
    assert rowops_device_status() == TIMEOUT
    assert rowops_device_status() == 0  # the status query clears the word
    # without the hook: same kernel, correct output, no error recorded
    monkeypatch.delenv("ROWOPS_TEST_STALL_ROW")
    y = rowops_softmax(x)
    assert rowops_device_status() == 0
    C.assert_softmax_close(C.to_f64(y), oracle.softmax(gu.rows_f32(x)), "bf16")


def test_layernorm_row_groups_wait_times_out(oracle, monkeypatch):
    wl = workloads.Workload("timeout_ln", "layernorm_gelu", "bf16", 1500, 8192, seed=4, affine=True)
    inp = gu.make_x(wl)
    monkeypatch.setenv("ROWOPS_KERNEL", "tma")
    monkeypatch.setenv("ROWOPS_WAIT_LIMIT_NS", LIMIT_NS)
    monkeypatch.setenv("ROWOPS_TEST_STALL_ROW", "3")
    rowops_layernorm_gelu(inp["x"], inp["w"], inp["b"], wl.eps)
    assert rowops_device_status() == TIMEOUT
    monkeypatch.delenv("ROWOPS_TEST_STALL_ROW")
    y = rowops_layernorm_gelu(inp["x"], inp["w"], inp["b"], wl.eps)
    assert rowops_device_status() == 0
    ref = oracle.layernorm_gelu(gu.rows_f32(inp["x"]), inp["w"].float().cpu().numpy(),
                                inp["b"].float().cpu().numpy(), wl.eps)
    C.assert_ln_gelu_close(C.to_f64(y), ref, "bf16")


def test_layernorm_flat_chunks_wait_times_out(oracle, monkeypatch):
    """The chunked kernel for short back-to-back rows: the copy of the chunk
    holding row 1000 never completes its phase."""
    wl = workloads.Workload("timeout_ln_flat", "layernorm_gelu", "bf16", 2001, 127, seed=6, affine=True)
    inp = gu.make_x(wl)
    monkeypatch.setenv("ROWOPS_KERNEL", "flat")
    monkeypatch.setenv("ROWOPS_WAIT_LIMIT_NS", LIMIT_NS)
    monkeypatch.setenv("ROWOPS_TEST_STALL_ROW", "1000")
    rowops_layernorm_gelu(inp["x"], inp["w"], inp["b"], wl.eps)
    assert rowops_device_status() == TIMEOUT
    monkeypatch.delenv("ROWOPS_TEST_STALL_ROW")
    y = rowops_layernorm_gelu(inp["x"], inp["w"], inp["b"], wl.eps)
    assert rowops_device_status() == 0
    ref = oracle.layernorm_gelu(gu.rows_f32(inp["x"]), inp["w"].float().cpu().numpy(),
                                inp["b"].float().cpu().numpy(), wl.eps)
    C.assert_ln_gelu_close(C.to_f64(y), ref, "bf16")


@pytest.mark.parametrize("staging", ["smem", "l2", "groups"])
def test_single_read_split_softmax_wait_times_out(oracle, monkeypatch, staging):
    wl = workloads.Workload("timeout_online", "online_softmax", "f32", 6, 1 << 20, seed=5)
    x = gu.make_x(wl)["x"]
    ws = torch.empty(rowops_online_softmax_workspace_bytes(6, 1 << 20, torch.float32), dtype=torch.uint8,
                     device="cuda")
    monkeypatch.setenv("ROWOPS_ONLINE", "row_groups" if staging == "groups" else "single_read")
    if staging == "l2":
        monkeypatch.setenv("ROWOPS_PERSIST_L2", "1")
    monkeypatch.setenv("ROWOPS_WAIT_LIMIT_NS", LIMIT_NS)
    monkeypatch.setenv("ROWOPS_TEST_STALL_ROW", "2")
    rowops_online_softmax(x, workspace=ws)
    assert rowops_online_softmax_status(ws) == TIMEOUT
    monkeypatch.delenv("ROWOPS_TEST_STALL_ROW")
    y = rowops_online_softmax(x, workspace=ws)
    assert rowops_online_softmax_status(ws) == 0
    C.assert_softmax_close(C.to_f64(y), oracle.softmax(gu.rows_f32(x)), "f32")


def test_two_pass_split_softmax_wait_times_out(oracle, monkeypatch):
    """The two-pass split softmax on full chunks streams them through a ring:
    a stalled chunk (work item 37) ends both passes' waits in a recorded
    timeout, reported through the workspace; the next call is correct."""
    wl = workloads.Workload("timeout_two_pass", "online_softmax", "f32", 4, 1 << 16, seed=6)
    x = gu.make_x(wl)["x"]
    ws = torch.empty(rowops_online_softmax_workspace_bytes(4, 1 << 16, torch.float32), dtype=torch.uint8,
                     device="cuda")
    monkeypatch.setenv("ROWOPS_WAIT_LIMIT_NS", LIMIT_NS)
    monkeypatch.setenv("ROWOPS_TEST_STALL_ROW", "37")
    rowops_online_softmax(x, workspace=ws, chunk=2048)
    assert rowops_online_softmax_status(ws) == TIMEOUT
    monkeypatch.delenv("ROWOPS_TEST_STALL_ROW")
    y = rowops_online_softmax(x, workspace=ws, chunk=2048)
    assert rowops_online_softmax_status(ws) == 0
    C.assert_softmax_close(C.to_f64(y), oracle.softmax(gu.rows_f32(x)), "f32")


@pytest.mark.parametrize("sched", ["static", "dynamic"])
def test_rmsnorm_pipeline_wait_times_out(oracle, monkeypatch, sched):
    """The fused residual RMSNorm ring (two input rows per slot on one
    mbarrier): the stalled row's wait gives up, the next call is correct.
    On the dynamic schedule the stalled group also drains a steal request it
    may have in flight."""
    from row_wise_reduction_gb300 import rowops_fused_residual_rmsnorm

    wl = workloads.Workload("timeout_rms", "residual_rmsnorm", "bf16", 1500, 8192, seed=6, affine=True,
                            residual=True)
    inp = gu.make_x(wl)
    monkeypatch.setenv("ROWOPS_KERNEL", "tma")
    monkeypatch.setenv("ROWOPS_SCHED", sched)
    monkeypatch.setenv("ROWOPS_WAIT_LIMIT_NS", LIMIT_NS)
    monkeypatch.setenv("ROWOPS_TEST_STALL_ROW", "11")
    rowops_fused_residual_rmsnorm(inp["x"], inp["residual"], inp["w"], wl.eps)
    assert rowops_device_status() == TIMEOUT
    monkeypatch.delenv("ROWOPS_TEST_STALL_ROW")
    y, ro = rowops_fused_residual_rmsnorm(inp["x"], inp["residual"], inp["w"], wl.eps)
    assert rowops_device_status() == 0
    s_ref, y_ref = oracle.residual_rmsnorm(gu.rows_f32(inp["x"]), gu.rows_f32(inp["residual"]),
                                           inp["w"].float().cpu().numpy(), wl.eps, "bf16")
    np.testing.assert_array_equal(C.to_f64(ro), s_ref)
    C.assert_rms_close(C.to_f64(y), y_ref, "bf16")


def test_causal_softmax_wait_times_out(oracle, monkeypatch):
    """The causal row pipeline (prefix copies): the stalled row's wait gives up."""
    from row_wise_reduction_gb300 import rowops_softmax_causal

    x = gu.make_x(_softmax_wl())["x"]
    monkeypatch.setenv("ROWOPS_KERNEL", "tma")
    monkeypatch.setenv("ROWOPS_WAIT_LIMIT_NS", LIMIT_NS)
    monkeypatch.setenv("ROWOPS_TEST_STALL_ROW", "1234")
    rowops_softmax_causal(x, 4096, 0)
    assert rowops_device_status() == TIMEOUT
    monkeypatch.delenv("ROWOPS_TEST_STALL_ROW")
    y = rowops_softmax_causal(x, 4096, 0)
    assert rowops_device_status() == 0
    C.assert_softmax_close(C.to_f64(y), oracle.softmax_causal(gu.rows_f32(x), 4096, 0), "bf16")


@pytest.mark.parametrize("partials", ["tmem", "registers"])
def test_layernorm_gelu_backward_wait_times_out(oracle, monkeypatch, partials):
    """The backward's ring (x and dy rows in one slot) gives up on the stalled
    row, records the timeout, and the next call is correct; with the partials
    in tensor memory the group that gave up leaves its row loop and the CTA
    still frees its tensor memory (the next call allocates it again)."""
    wl = workloads.Workload("timeout_ln_bwd", "layernorm_gelu_backward", "bf16", 1200, 8192, seed=4, affine=True,
                            grad=True)
    inp = gu.make_x(wl)
    monkeypatch.setenv("ROWOPS_KERNEL", "tma")
    monkeypatch.setenv("ROWOPS_BWD_PARTIALS", partials)
    monkeypatch.setenv("ROWOPS_WAIT_LIMIT_NS", LIMIT_NS)
    monkeypatch.setenv("ROWOPS_TEST_STALL_ROW", "400")
    rowops_layernorm_gelu_backward(inp["x"], inp["dy"], inp["w"], inp["b"], wl.eps)
    assert rowops_device_status() == TIMEOUT
    monkeypatch.delenv("ROWOPS_TEST_STALL_ROW")
    dx, dw, db = rowops_layernorm_gelu_backward(inp["x"], inp["dy"], inp["w"], inp["b"], wl.eps)
    assert rowops_device_status() == 0
    rows = gu.sample_rows(wl.M, 8)
    ref_dx, _, _ = oracle.layernorm_gelu_backward(gu.rows_f32(inp["x"], rows), gu.rows_f32(inp["dy"], rows),
                                                  inp["w"].float().cpu().numpy(), inp["b"].float().cpu().numpy(),
                                                  wl.eps)
    got = C.to_f64(dx[torch.as_tensor(rows, device=dx.device)])
    assert np.all(np.abs(got - ref_dx) <= C.bf16_ulp(ref_dx) + 1e-3)
