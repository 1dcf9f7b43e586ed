"""Host-side logic of bench.py that needs no GPU: the multi-rank aggregation
(max time, summed work) over two gloo ranks on the CPU, the reference arm's
rank-0-only rule, and the byte accounting."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        secs, units = bench.aggregate(0.5 + rank, 100.0 * (rank + 1))
        q.put((rank, secs, units))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, secs, units in got:
        assert secs == 1.5  # the slowest rank's time
        assert units == 300.0  # every rank's work


def test_aggregate_without_process_group_is_identity():
    import bench

    assert bench.aggregate(2.0, 7.0) == (2.0, 7.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""


def test_algorithmic_bytes():
    import bench
    from row_wise_reduction_gb300 import workloads

    W = workloads.WORKLOADS
    assert bench.alg_bytes(W["softmax_bf16_causal_32768x4096"]) == 2 * 32768 * 4096 * 2
    assert bench.alg_bytes(W["online_softmax_f32_64x1048576"]) == 2 * 64 * (1 << 20) * 4
    assert bench.alg_bytes(W["layernorm_gelu_bf16_65536x8192"]) == 2 * 65536 * 8192 * 2 + 2 * 8192 * 2


def test_profiled_traffic_requires_matching_source(tmp_path, monkeypatch):
    import bench

    p = tmp_path / "summary.txt"
    p.write_text(f"kernel_source_sha: {bench.dominant_source_hash()}\ndram_bytes_per_launch: 123\n")
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(p))
    assert bench.profiled_traffic() == 123
    p.write_text("kernel_source_sha: 0000\ndram_bytes_per_launch: 123\n")
    assert bench.profiled_traffic() is None


def test_kernel_count_without_gpu_activity_falls_back():
    """With no CUDA activity in the trace (no GPU here, or nothing launched)
    the profiler count is None, so the bench uses its per-operation table."""
    import bench
    assert bench.count_kernels(lambda: None) is None
    assert set(bench.KERNELS_PER_CALL) >= {"softmax_causal", "online_softmax", "layernorm_gelu"}


def test_fractions_of_the_three_ceilings():
    """The bench line reports one rate against the measured peak, the
    copy measured in the same run and nominal HBM; a missing in-run copy gives
    no fraction rather than a wrong one."""
    import bench

    f = bench.fractions(6000.0, 6690.5, 6500.0)
    assert f["frac"] == 6000.0 / 6690.5
    assert f["frac_of_in_run_copy"] == 6000.0 / 6500.0
    assert f["frac_of_nominal"] == 6000.0 / bench.NOMINAL_HBM_GBS == 0.75
    assert bench.fractions(6000.0, 6690.5, None)["frac_of_in_run_copy"] is None


def test_host_link_ceiling_arithmetic():
    """The end-to-end ceiling is the step's algorithmic bytes over the time of
    the copy-only pipeline: 3.22 GB per step, 5 steps in 50 ms -> 322 GB/s."""
    import bench

    step = sum(bench.alg_bytes(bench.workloads.WORKLOADS[n]) for n in bench.STEP)
    assert step == 3221258240
    assert abs(bench.link_ceiling(step, 0.050, 5) - step * 5 / 0.050 / 1e9) < 1e-9
    assert abs(bench.link_ceiling(step, 0.050, 5) - 322.125824) < 1e-6


def test_step_dtype_label_names_both_io_types():
    """The step computes in fp32 with bf16 and fp32 inputs and outputs; the
    label says so instead of a single type."""
    import bench
    from row_wise_reduction_gb300 import workloads

    io = {workloads.WORKLOADS[n].dtype for n in bench.STEP}
    assert io == {"bf16", "f32"}
    assert bench.STEP_DTYPE.startswith("f32 arithmetic")
    assert "bf16" in bench.STEP_DTYPE and "f32 I/O" in bench.STEP_DTYPE


def test_row_blocks_of_a_larger_problem():
    """Under torchrun rank r draws rows [r M, (r + 1) M) of the workload's
    (world M)-row problem: its own data, the causal mask of its global row
    indices, the problem's w and b."""
    import torch
    from row_wise_reduction_gb300 import workloads

    wl = workloads.Workload("blk", "softmax_causal", "f32", 6, 4, seed=3, causal=True)
    b0 = workloads.make_inputs(wl, "cpu", block=0)["x"]
    b1 = workloads.make_inputs(wl, "cpu", block=1)["x"]
    kept = lambda x: (~torch.isinf(x)).sum(dim=1).tolist()  # noqa: E731
    assert kept(b0) == [1, 2, 3, 4, 1, 2]  # rows 0..5: r mod 4 + 1 columns
    assert kept(b1) == [3, 4, 1, 2, 3, 4]  # rows 6..11
    assert not torch.equal(b0[:, 0], b1[:, 0])
    aff = workloads.Workload("blk_ln", "layernorm_gelu", "f32", 3, 8, seed=5, affine=True)
    a0, a1 = workloads.make_inputs(aff, "cpu", block=0), workloads.make_inputs(aff, "cpu", block=2)
    assert torch.equal(a0["w"], a1["w"]) and torch.equal(a0["b"], a1["b"])
    assert not torch.equal(a0["x"], a1["x"])
    assert torch.equal(workloads.make_inputs(aff, "cpu")["x"], a0["x"])  # block 0 is the one-GPU workload
