#!/usr/bin/env python
"""Benchmark of the row-wise reduce-then-normalise path on GB300.

One step runs the whole hot path once, each operation on its full-size
synthetic workload:
  * rowops_softmax          bf16 32768 x 4096, causal -inf mask   (537 MB moved)
  * rowops_online_softmax   fp32 64 x 2^20, +30 outliers          (537 MB moved)
  * rowops_layernorm_gelu   bf16 65536 x 8192, w, b               (2148 MB moved)
and ``value`` is the algorithmic HBM bytes of a step (each input read once,
each output written once) times the steps, over the device time of the timed
steps: GB/s. Each input is larger than the 129 MB L2, so no flush is needed
between steps. The roofline entry is the dominant kernel (LayerNorm+GELU)
against the measured copy bandwidth (MEASURED_PEAKS.json), with its
fractions of a device-to-device copy timed in this same process and of the
8 TB/s nominal HBM figure beside it. ``e2e`` repeats the step through the
public API with pinned host buffers (inputs copied in and results copied out
inside the timed region) and carries the host link's own ceiling, timed in the
same run: the same copy pipeline with no kernel.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl rowops|reference]

Under torchrun rank r takes the contiguous row block [r M, (r + 1) M) of each
workload's (world M)-row problem (weak scaling, no collective on the data
path); rank 0 prints one JSON line.
``--impl reference`` times the double-precision CPU oracle on host cores on a
bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from row_wise_reduction_gb300 import workloads  # noqa: E402

METRIC = "row-kernel HBM GB/s (% of GB300 peak) for softmax and LayerNorm+GELU"
STEP = ["softmax_bf16_causal_32768x4096", "online_softmax_f32_64x1048576", "layernorm_gelu_bf16_65536x8192"]
DOMINANT = "layernorm_gelu_bf16_65536x8192"
# kernels per call, the fallback when the profiler cannot count them (the
# online softmax at these sizes: one cooperative kernel, no memset)
KERNELS_PER_CALL = {"softmax": 1, "softmax_causal": 1, "online_softmax": 1, "layernorm_gelu": 1,
                    "layernorm_gelu_erf": 1, "rmsnorm": 1, "residual_rmsnorm": 1, "row_sum": 1, "row_max": 1,
                    "layernorm_gelu_backward": 2, "bias_residual_gelu": 1}
L2_BYTES = 129 * 10**6
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # the HBM figure the hardware table gives for this class of GPU
COPY_PROBE_BYTES = 1 << 30  # the in-run device-to-device copy: 1 GiB, read + write counted
# arithmetic type of the step (every operation accumulates in fp32) and the I/O types
STEP_DTYPE = "f32 arithmetic; bf16 I/O (softmax, LayerNorm+GELU), f32 I/O (online softmax)"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "ln_gelu_bf16_65536x8192.txt")
DOMINANT_SOURCES = ["row_wise_reduction_gb300/csrc/tma_row_kernels.cuh",
                    "row_wise_reduction_gb300/csrc/row_pipeline.cuh",
                    "row_wise_reduction_gb300/csrc/tma_inst.cuh",
                    "row_wise_reduction_gb300/csrc/ln_gelu_kernels.cuh",
                    "row_wise_reduction_gb300/csrc/rowops_device.cuh",
                    "row_wise_reduction_gb300/csrc/rowops_launch.h"]


def alg_bytes(wl: workloads.Workload) -> int:
    """Each input element read once, each output element written once, w (and
    b) once per launch."""
    es = workloads.elem_size(wl.dtype)
    rows = 2 * wl.M * wl.N * es
    if wl.op in ("layernorm_gelu", "layernorm_gelu_erf"):
        return rows + (2 * wl.N * es if wl.affine else 0)
    if wl.op in ("row_sum", "row_max"):  # x read, one fp32 per row written
        return wl.M * wl.N * es + wl.M * 4
    if wl.op == "rmsnorm":
        return rows + (wl.N * es if wl.affine else 0)
    if wl.op == "residual_rmsnorm":  # x, residual in; y, residual_out out
        return 2 * rows + (wl.N * es if wl.affine else 0)
    if wl.op == "softmax_causal":  # kept entries read, every output written
        return causal_alg_bytes(wl, wl.N)
    if wl.op == "bias_residual_gelu":  # x, residual in; y out; the bias once
        return 3 * wl.M * wl.N * es + wl.N * es
    if wl.op == "layernorm_gelu_backward":  # x, dy in; dx out; w, b in; fp32 dw, db out
        return 3 * wl.M * wl.N * es + (2 * wl.N * es if wl.affine else 0) + 2 * wl.N * 4
    return rows


def fractions(achieved: float, peak: float, in_run_copy, nominal: float = NOMINAL_HBM_GBS) -> dict:
    """The achieved rate as a fraction of the measured peak, of the copy
    ceiling measured in the same run (None when not measured) and of nominal."""
    return {"frac": achieved / peak,
            "frac_of_in_run_copy": achieved / in_run_copy if in_run_copy else None,
            "frac_of_nominal": achieved / nominal}


def link_ceiling(step_bytes: int, copies_only_s: float, steps: int) -> float:
    """The end-to-end figure the host link allows: the step's algorithmic bytes
    over the time of the same pipeline with the copies and without the
    kernels (GB/s)."""
    return step_bytes * steps / copies_only_s / 1e9


def dominant_source_hash() -> str:
    h = hashlib.sha256()
    for p in DOMINANT_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if that summary was taken on the current kernel source."""
    try:
        kv = {}
        with open(PROFILE_SUMMARY) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha") != dominant_source_hash():
            return None
        return int(float(kv["dram_bytes_per_launch"]))
    except (OSError, KeyError, ValueError):
        return None


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region: NVML through ctypes (read-only queries),
# nvidia-smi as a fallback
# ---------------------------------------------------------------------------
REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
           0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
           0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}


class ClockSampler:
    def __init__(self, device: int, period_s: float = 0.001):
        self.period = period_s
        self.samples = []
        self.max_mhz = None
        self.src = None
        self._stop = threading.Event()
        self._thread = None
        self._smi = None
        self._smi_out = None
        self.uuid = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(device).uuid)
            if not self.uuid.startswith("GPU-"):
                self.uuid = "GPU-" + self.uuid
        except Exception:
            self.uuid = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            if self.uuid is None or nv.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
            v = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(v)) == 0:
                self.max_mhz = v.value
            self._nv, self._h = nv, h
            self._reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.src = "nvml"
        except Exception:
            self._nv = None

    def _poll(self):
        nv, h = self._nv, self._h
        clk, rs, pw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                r = rs.value if self._reasons(h, ctypes.byref(rs)) == 0 else 0
                p = pw.value / 1000.0 if nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0 else None
                self.samples.append((clk.value, r, p))
            time.sleep(self.period)

    def start(self, csv_path=None):
        if self._nv is not None:
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
        if csv_path:
            q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
            cmd = ["nvidia-smi", f"--query-gpu={q}", "--format=csv", "-lms", "200"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            try:
                self._smi_out = open(csv_path, "w")
                self._smi = subprocess.Popen(cmd, stdout=self._smi_out, stderr=subprocess.DEVNULL)
            except OSError:
                self._smi = None

    def stop(self):
        self._stop.set()
        if self._thread:
            self._thread.join()
        if self._smi:
            self._smi.terminate()
            self._smi.wait()
            self._smi_out.close()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0, "source": self.src}
        mhz = [s[0] for s in self.samples]
        bits = 0
        for s in self.samples:
            bits |= s[1]
        reasons = [name for bit, name in REASONS.items() if bits & bit and name != "gpu_idle"]
        power = [s[2] for s in self.samples if s[2] is not None]
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(mhz), "power_w_max": max(power) if power else None, "source": self.src}


def copy_ceiling(dev, reps: int = 10, nbytes: int = COPY_PROBE_BYTES):
    """Device-to-device copy of `nbytes` (cudaMemcpyAsync through torch's
    copy_ of same-dtype contiguous tensors), best of `reps` by CUDA events;
    GB/s counting bytes read + written. Measured in this process, next to the
    kernels it is the ceiling for."""
    a = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    b = torch.empty_like(a)
    a.fill_(1)
    stream = torch.cuda.current_stream()
    best = float("inf")
    for _ in range(reps + 2):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        b.copy_(a)
        e1.record(stream)
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) / 1e3)
    del a, b
    torch.cuda.empty_cache()
    return 2 * nbytes / best / 1e9


HOST_COST_DRIVER = os.path.join(ROOT, "tests", "native", "host_cost.c")


def host_cost_c(timeout_s: float = 120.0):
    """Per-call host cost of rowops_softmax measured from C (no Python layer):
    compiles the small driver against librowops.so and the CUDA runtime, runs
    it and returns its JSON result, or None when no compiler or GPU is there."""
    import shutil
    import tempfile

    from row_wise_reduction_gb300 import build as rbuild

    cc = shutil.which("gcc") or shutil.which("cc")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    if cc is None or not os.path.exists(rbuild.LIB):
        return None
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "host_cost")
        libdir = os.path.dirname(rbuild.LIB)
        cmd = [cc, "-O2", "-std=c11", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
               HOST_COST_DRIVER, "-o", exe, "-L", libdir, "-l:librowops.so", "-L", os.path.join(cuda, "lib64"),
               "-lcudart", f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
        if subprocess.run(cmd, capture_output=True, text=True).returncode != 0:
            return None
        r = subprocess.run([exe], capture_output=True, text=True, timeout=timeout_s)
        if r.returncode != 0:
            return None
        return json.loads(r.stdout.strip().splitlines()[-1])


def host_cost_python(dev, batch: int = 256, batches: int = 20):
    """The same measurement through the Python binding: wall time of issuing
    rowops_softmax(x, y) on fp32 1024 x 768, per call (each batch timed while
    issuing, then synchronised); the median over the batches, so that a batch
    disturbed by other host work does not set the figure."""
    import row_wise_reduction_gb300 as ro

    x = torch.randn(1024, 768, device=dev)
    y = torch.empty_like(x)
    for _ in range(200):
        ro.rowops_softmax(x, y)
    torch.cuda.synchronize()
    per_call = []
    for _ in range(batches):
        t0 = time.perf_counter()
        for _ in range(batch):
            ro.rowops_softmax(x, y)
        per_call.append((time.perf_counter() - t0) / batch * 1e6)
        torch.cuda.synchronize()
    return statistics.median(per_call)


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU, launched by torchrun)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def count_kernels(fn):
    """Kernels that one call of fn launches, from the profiler's CUDA activity
    trace (memsets and copies excluded); None if no activity was recorded."""
    try:
        from torch.profiler import ProfilerActivity, profile
        torch.cuda.synchronize()
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            fn()
            torch.cuda.synchronize()
        kinds = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]
    except Exception:
        return None
    kernels = [k for k in kinds if not k.startswith(("Memset", "Memcpy", "cudaMemset", "cudaMemcpy"))]
    return len(kernels) if kernels else None


def aggregate(seconds: float, units: float, group=None):
    """Max of the per-rank times and sum of the per-rank work over the process
    group (identity without one)."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return seconds, units
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# the CPU oracle on a bounded sample
# ---------------------------------------------------------------------------
def oracle_run(oracle, wl, xs, extra, lo=0, hi=None):
    """The oracle's version of ``wl``'s operation on sampled rows xs (rows
    lo:hi of the sample; per-row inputs and row indices in ``extra``)."""
    hi = len(xs) if hi is None else hi
    xs = xs[lo:hi]
    per_row = {k: extra[k][lo:hi] for k in ("residual", "dy") if extra.get(k) is not None}
    w, b = extra.get("w"), extra.get("b")
    if wl.op == "softmax":
        oracle.softmax(xs)
    elif wl.op == "online_softmax":
        oracle.split_softmax(xs, extra["chunk"])
    elif wl.op == "softmax_causal":
        for x, r in zip(xs, extra["rows"][lo:hi]):
            oracle.softmax_causal_rows_at(x, int(r), wl.N, 0)
    elif wl.op in ("row_sum", "row_max"):
        getattr(oracle, wl.op)(xs)
    elif wl.op == "rmsnorm":
        oracle.rmsnorm(xs, w, wl.eps)
    elif wl.op == "residual_rmsnorm":
        oracle.residual_rmsnorm(xs, per_row["residual"], w, wl.eps, storage=wl.dtype)
    elif wl.op == "layernorm_gelu_erf":
        oracle.layernorm_gelu_erf(xs, w, b, wl.eps)
    elif wl.op == "layernorm_gelu_backward":
        oracle.layernorm_gelu_backward(xs, per_row["dy"], w, b, wl.eps)
    elif wl.op == "bias_residual_gelu":
        oracle.bias_residual_gelu(xs, per_row["residual"], b)
    else:
        oracle.layernorm_gelu(xs, w, b, wl.eps)


def oracle_run_threads(oracle, wl, xs, extra, threads):
    """The oracle on contiguous row slices in `threads` host threads (ctypes
    releases the GIL inside the C calls, so the slices run on separate cores)."""
    if threads <= 1 or len(xs) < 2:
        oracle_run(oracle, wl, xs, extra)
        return
    from concurrent.futures import ThreadPoolExecutor

    bounds = [len(xs) * i // threads for i in range(threads + 1)]
    spans = [(a, b) for a, b in zip(bounds, bounds[1:]) if b > a]
    with ThreadPoolExecutor(len(spans)) as ex:
        list(ex.map(lambda ab: oracle_run(oracle, wl, xs, extra, *ab), spans))


def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_sample_rows(wl, rows, device=None, dev_inputs=None):
    """fp32 host rows of ``wl`` (copied from the device inputs when given,
    else drawn on the CPU with the causal mask of rows spread over the
    workload) plus w, b, the same rows of the residual / dy where the
    operation has them, and the row indices."""
    import numpy as np

    if dev_inputs is not None:
        idx = torch.as_tensor(rows, device=dev_inputs["x"].device)
        src = dev_inputs
    else:
        idx = None
        src = workloads.make_inputs(wl.with_shape(M=len(rows)), "cpu", row_ids=torch.as_tensor(rows))
    pick = (lambda t: t[idx]) if idx is not None else (lambda t: t)
    xs = pick(src["x"]).float().cpu().numpy()
    extra = {k: src[k].float().cpu().numpy() for k in ("w", "b") if k in src}
    for k in ("residual", "dy"):
        if k in src:
            extra[k] = np.ascontiguousarray(pick(src[k]).float().cpu().numpy())
    extra.setdefault("w", None)
    extra.setdefault("b", None)
    extra["chunk"] = 8192
    extra["rows"] = list(rows)
    return np.ascontiguousarray(xs), extra


def spread_rows(M, k):
    if k >= M:
        return list(range(M))
    step = M / k
    return [int(i * step) for i in range(k)]


def cpu_baseline(oracle, dev_inputs=None, budget_s=12.0, threads=1, wls=None):
    """Time the oracle on ~budget_s seconds (wall) of the timed workloads
    (`wls`, name -> Workload; default the step's) in `threads` host threads;
    return GB/s on the same algorithmic-byte basis, a description of the
    sample and the seconds spent."""
    wls = wls or {n: workloads.WORKLOADS[n] for n in STEP}
    total_bytes, total_s, desc = 0, 0.0, []
    per_op = budget_s / len(wls)
    for name, wl in wls.items():
        # calibrate on one row, then size the sample to the budget
        xs, extra = cpu_sample_rows(wl, [wl.M // 2], dev_inputs=dev_inputs.get(name) if dev_inputs else None)
        t0 = time.perf_counter()
        oracle_run(oracle, wl, xs, extra)
        dt = max(time.perf_counter() - t0, 1e-6)
        k = max(1, min(wl.M, int(per_op * threads / dt)))
        rows = spread_rows(wl.M, k)
        xs, extra = cpu_sample_rows(wl, rows, dev_inputs=dev_inputs.get(name) if dev_inputs else None)
        t0 = time.perf_counter()
        oracle_run_threads(oracle, wl, xs, extra, threads)
        total_s += time.perf_counter() - t0
        total_bytes += alg_bytes(wl.with_shape(M=len(rows)))
        desc.append(f"{len(rows)} of {wl.M} rows of {name}")
    return total_bytes / total_s / 1e9, "; ".join(desc), total_s


# ---------------------------------------------------------------------------
# reference arm: the oracle on host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from oracle import oracle

    oracle.build()
    K, W = args.steps, args.warmup
    threads = host_threads()
    per_step_s = max(0.3, min(3.0, args.reference_budget_s / max(1, K + W)))
    # calibrate rows per op on one row each
    samples = []
    for name in STEP:
        wl = workloads.WORKLOADS[name]
        xs, extra = cpu_sample_rows(wl, [wl.M // 2])
        t0 = time.perf_counter()
        oracle_run(oracle, wl, xs, extra)
        dt = max(time.perf_counter() - t0, 1e-6)
        k = max(1, min(wl.M, int(per_step_s * threads / len(STEP) / dt)))
        rows = spread_rows(wl.M, k)
        samples.append((wl, *cpu_sample_rows(wl, rows), len(rows)))
    step_bytes = sum(alg_bytes(wl.with_shape(M=k)) for wl, _, _, k in samples)

    def step():
        for wl, xs, extra, _ in samples:
            oracle_run_threads(oracle, wl, xs, extra, threads)

    for _ in range(W):
        step()
    t0 = time.perf_counter()
    for _ in range(K):
        step()
    secs = time.perf_counter() - t0
    value = step_bytes * K / secs / 1e9
    sample = "; ".join(f"{k} of {wl.M} rows of {wl.name}" for wl, _, _, k in samples) + " per step"
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": secs / K * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": config_block(),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


def parallelism(world: int) -> str:
    if world == 1:
        return "one GPU"
    return (f"row blocks: rank r takes rows [r M, (r + 1) M) of each workload's {world} M-row problem; "
            "no collective on the data path")


def config_block(world: int = 1):
    return {
        "workload": " + ".join(STEP),
        "parallelism": parallelism(world),
        "per_step_bytes": {n: alg_bytes(workloads.WORKLOADS[n]) for n in STEP},
        "l2": "no flush: every input (268 MB, 268 MB, 1074 MB) is larger than the 129 MB L2",
        "bytes_basis": "algorithmic: each input element read once, each output element written once (+ w, b)",
    }


# ---------------------------------------------------------------------------
# the other workloads, reported beside the step (not part of its value)
# ---------------------------------------------------------------------------
def causal_alg_bytes(wl: workloads.Workload, period: int, offset: int = 0) -> int:
    """Kept entries read once, every output element written once."""
    import numpy as np

    r = np.arange(wl.M)
    kept = np.clip(r % period + offset + 1, 0, wl.N)
    es = workloads.elem_size(wl.dtype)
    return int(kept.sum()) * es + wl.M * wl.N * es


EXTRA = ["softmax_f32_1024x768", "layernorm_gelu_f32_4096x768", "layernorm_gelu_bf16_65536x127",
         "layernorm_gelu_bf16_65536x4097", "rmsnorm_f32_4096x768", "residual_rmsnorm_f32_4096x768",
         "rmsnorm_bf16_65536x8192", "residual_rmsnorm_bf16_65536x8192", "softmax_causal_bf16_32768x4096",
         "layernorm_gelu_erf_f32_4096x768", "layernorm_gelu_erf_bf16_65536x8192", "row_sum_bf16_65536x8192",
         "row_max_bf16_65536x8192", "layernorm_gelu_backward_f32_4096x768",
         "layernorm_gelu_backward_bf16_65536x8192", "bias_residual_gelu_f32_4096x768",
         "bias_residual_gelu_bf16_65536x8192"]
SMALL = {"softmax_f32_1024x768", "layernorm_gelu_f32_4096x768", "rmsnorm_f32_4096x768",
         "residual_rmsnorm_f32_4096x768", "layernorm_gelu_erf_f32_4096x768", "layernorm_gelu_backward_f32_4096x768",
         "bias_residual_gelu_f32_4096x768"}


def run_extras(dev, stream, iters=50):
    """Per workload: the kernel time with inputs hot in L2 (back to back), with
    L2 flushed before each launch (a 512 MB write between launches, outside the
    timed events), and per launch inside a CUDA graph of `iters` launches."""
    import row_wise_reduction_gb300 as ro

    flush = torch.empty(512 * 2**20, dtype=torch.uint8, device=dev)
    out = {}
    for name in EXTRA:
        wl = workloads.WORKLOADS[name]
        inp = workloads.make_inputs(wl, dev)
        x, y = inp["x"], torch.empty_like(inp["x"])
        r_out = torch.empty_like(x) if wl.residual else None
        red = torch.empty(wl.M, dtype=torch.float32, device=dev)
        if wl.grad:
            dw = torch.empty(wl.N, dtype=torch.float32, device=dev)
            db = torch.empty(wl.N, dtype=torch.float32, device=dev)
            ws = torch.empty(ro.rowops_layernorm_gelu_backward_workspace_bytes(wl.M, wl.N, x.dtype),
                             dtype=torch.uint8, device=dev)

        def call():
            if wl.op == "layernorm_gelu_backward":
                ro.rowops_layernorm_gelu_backward(x, inp["dy"], inp.get("w"), inp.get("b"), wl.eps, y, dw, db, ws)
            elif wl.op == "bias_residual_gelu":
                ro.rowops_bias_residual_gelu(x, inp["residual"], inp["b"], y)
            elif wl.op == "softmax":
                ro.rowops_softmax(x, y)
            elif wl.op == "row_sum":
                ro.rowops_row_sum(x, red)
            elif wl.op == "row_max":
                ro.rowops_row_max(x, red)
            elif wl.op == "layernorm_gelu_erf":
                ro.rowops_layernorm_gelu_erf(x, inp.get("w"), inp.get("b"), wl.eps, y)
            elif wl.op == "softmax_causal":
                ro.rowops_softmax_causal(x, wl.N, 0, y)
            elif wl.op == "rmsnorm":
                ro.rowops_rmsnorm(x, inp.get("w"), wl.eps, y)
            elif wl.op == "residual_rmsnorm":
                ro.rowops_fused_residual_rmsnorm(x, inp["residual"], inp.get("w"), wl.eps, y, r_out)
            else:
                ro.rowops_layernorm_gelu(x, inp.get("w"), inp.get("b"), wl.eps, y)

        for _ in range(5):
            call()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(iters):
            call()
        b.record(stream)
        torch.cuda.synchronize()
        hot = a.elapsed_time(b) / iters / 1e3
        rec = {"bytes": alg_bytes(wl), "hot_us": hot * 1e6, "hot_gbs": alg_bytes(wl) / hot / 1e9,
               "hot_rows_per_s": wl.M / hot}
        if alg_bytes(wl) > L2_BYTES:
            rec["frac_of_" + measured_peak()[1]] = rec["hot_gbs"] / measured_peak()[0]
        if wl.op in ("rmsnorm", "residual_rmsnorm", "layernorm_gelu_backward", "bias_residual_gelu") and \
                wl.M * wl.N > 10**6:
            rec["torch_eager"] = torch_eager_time(wl, inp, stream)
        if name in SMALL:
            cold = []
            for _ in range(10):
                flush.fill_(1)
                a.record(stream)
                call()
                b.record(stream)
                torch.cuda.synchronize()
                cold.append(a.elapsed_time(b) / 1e3)
            c = statistics.median(cold)
            rec.update(cold_us=c * 1e6, cold_gbs=alg_bytes(wl) / c / 1e9)
            g = torch.cuda.CUDAGraph()
            s2 = torch.cuda.Stream()
            s2.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s2):
                call()
                torch.cuda.synchronize()
                with torch.cuda.graph(g, stream=s2):
                    for _ in range(iters):
                        call()
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            gt = a.elapsed_time(b) / iters / 1e3
            rec.update(graph_us=gt * 1e6, graph_gbs=alg_bytes(wl) / gt / 1e9, l2_resident=True)
        out[name] = rec
        del inp, x, y, r_out, red
    del flush
    return out


def torch_eager_time(wl, inp, stream, iters=10):
    """PyTorch eager as context: on an RMSNorm workload F.rms_norm, and for the
    fused form x + residual followed by F.rms_norm (two kernels at least); on
    the backward workload autograd's gradients of gelu(layer_norm(x)) (tanh)
    for x, w, b from a retained graph (the backward kernels only); on the fused
    residual + bias + GELU workload F.gelu(x + b + residual) (three kernels)."""
    import torch.nn.functional as F

    x, w = inp["x"], inp.get("w")
    if wl.op == "bias_residual_gelu":
        r, bias = inp["residual"], inp["b"]

        def call():
            return F.gelu(x + bias + r)
        what = "F.gelu(x + b + residual)"
    elif wl.op == "layernorm_gelu_backward":
        xg = x.detach().clone().requires_grad_(True)
        wg = w.detach().clone().requires_grad_(True)
        bg = inp["b"].detach().clone().requires_grad_(True)
        out = F.gelu(F.layer_norm(xg, (wl.N,), wg, bg, wl.eps), approximate="tanh")
        dy = inp["dy"]

        def call():
            return torch.autograd.grad(out, (xg, wg, bg), dy, retain_graph=True)
        what = "torch.autograd.grad(gelu(layer_norm(x, w, b), 'tanh'), (x, w, b), dy)"
    elif wl.op == "rmsnorm":
        def call():
            return F.rms_norm(x, (wl.N,), w, wl.eps)
        what = "F.rms_norm(x, (N,), w, eps)"
    else:
        r = inp["residual"]

        def call():
            s = x + r
            return F.rms_norm(s, (wl.N,), w, wl.eps), s
        what = "s = x + residual; F.rms_norm(s, (N,), w, eps)"
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(iters):
        call()
    b.record(stream)
    torch.cuda.synchronize()
    t = a.elapsed_time(b) / iters / 1e3
    return {"call": what, "us": t * 1e6, "gbs": alg_bytes(wl) / t / 1e9}


def run_torch_eager(wls, inputs, stream, iters=10):
    """PyTorch's own eager kernels on the step's workloads, as context: softmax
    along rows, and gelu(layer_norm(x)) unfused (tanh form). GB/s on the same
    algorithmic bytes as the step (the unfused pair moves more than that)."""
    import torch.nn.functional as F

    out = {}
    for n, wl in wls.items():
        x = inputs[n]["x"]
        if wl.op in ("softmax", "online_softmax"):
            def call():
                return torch.softmax(x, dim=-1)
            what = "torch.softmax(x, dim=-1)"
        else:
            w, b = inputs[n]["w"], inputs[n]["b"]

            def call():
                return F.gelu(F.layer_norm(x, (wl.N,), w, b, wl.eps), approximate="tanh")
            what = "F.gelu(F.layer_norm(x, (N,), w, b, eps), approximate='tanh')"
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(iters):
            call()
        b_.record(stream)
        torch.cuda.synchronize()
        t = a.elapsed_time(b_) / iters / 1e3
        out[n] = {"call": what, "avg_ms": t * 1e3, "gbs": alg_bytes(wl) / t / 1e9}
    return out


# ---------------------------------------------------------------------------
# rowops arm
# ---------------------------------------------------------------------------
def run_rowops(args):
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        print(json.dumps({"error": "bench.py needs a CUDA GPU"}))
        return 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    import row_wise_reduction_gb300 as ro

    ro.library()
    K, W = args.steps, args.warmup
    keys = {"softmax": STEP[0], "online": STEP[1], "layernorm": STEP[2]}
    if args.workloads:
        names = args.workloads.split(",")
        unknown = [n for n in names if n not in workloads.WORKLOADS]
        if unknown:
            raise SystemExit(f"unknown workloads {unknown}; known: {sorted(workloads.WORKLOADS)}")
    else:
        names = [keys[o] for o in args.ops.split(",")] if args.ops else list(STEP)
    subset = bool(args.ops or args.workloads)
    wls = {n: workloads.WORKLOADS[n] for n in names}
    if args.rows_scale != 1.0:
        wls = {n: wl.with_shape(M=max(1, int(wl.M * args.rows_scale))) for n, wl in wls.items()}
    inputs, outputs, ws = {}, {}, {}
    for n, wl in wls.items():
        # rank r: the contiguous row block [r M, (r + 1) M) of a (world M)-row problem
        inputs[n] = workloads.make_inputs(wl, dev, block=rank)
        outputs[n] = torch.empty_like(inputs[n]["x"])
        if wl.op == "online_softmax":
            nb = ro.rowops_online_softmax_workspace_bytes(wl.M, wl.N, workloads.torch_dtype(wl.dtype))
            ws[n] = torch.empty(nb, dtype=torch.uint8, device=dev)
        if wl.op == "layernorm_gelu_backward":
            nb = ro.rowops_layernorm_gelu_backward_workspace_bytes(wl.M, wl.N, workloads.torch_dtype(wl.dtype))
            ws[n] = (torch.empty(nb, dtype=torch.uint8, device=dev), torch.empty(wl.N, device=dev),
                     torch.empty(wl.N, device=dev))
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    res_out = {n: torch.empty_like(inputs[n]["x"]) for n, wl in wls.items() if wl.residual}
    reds = {n: torch.empty(wl.M, dtype=torch.float32, device=dev) for n, wl in wls.items()
            if wl.op in ("row_sum", "row_max")}

    def call(n, x, y):
        wl = wls[n]
        if wl.op == "softmax":
            ro.rowops_softmax(x, y)
        elif wl.op == "softmax_causal":
            ro.rowops_softmax_causal(x, wl.N, 0, y)
        elif wl.op == "row_sum":
            ro.rowops_row_sum(x, reds[n])
        elif wl.op == "row_max":
            ro.rowops_row_max(x, reds[n])
        elif wl.op == "layernorm_gelu_erf":
            ro.rowops_layernorm_gelu_erf(x, inputs[n]["w"], inputs[n]["b"], wl.eps, y)
        elif wl.op == "online_softmax":
            ro.rowops_online_softmax(x, y, workspace=ws[n])
        elif wl.op == "rmsnorm":
            ro.rowops_rmsnorm(x, inputs[n]["w"], wl.eps, y)
        elif wl.op == "residual_rmsnorm":
            ro.rowops_fused_residual_rmsnorm(x, inputs[n]["residual"], inputs[n]["w"], wl.eps, y, res_out[n])
        elif wl.op == "bias_residual_gelu":
            ro.rowops_bias_residual_gelu(x, inputs[n]["residual"], inputs[n]["b"], y)
        elif wl.op == "layernorm_gelu_backward":
            wsb, dw, db = ws[n]
            ro.rowops_layernorm_gelu_backward(x, inputs[n]["dy"], inputs[n]["w"], inputs[n]["b"], wl.eps, y, dw, db,
                                              wsb)
        else:
            ro.rowops_layernorm_gelu(x, inputs[n]["w"], inputs[n]["b"], wl.eps, y)

    # warm-up
    for _ in range(W):
        for n in names:
            call(n, inputs[n]["x"], outputs[n])
    torch.cuda.synchronize()
    # the device-to-device copy ceiling, measured in this process before the timed region
    copy_gbs = copy_ceiling(dev)

    # timed region: K steps, per-operation events on the launching stream
    ev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
          for n in names}
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start(args.clocks_csv if rank == 0 else None)
    t_start.record(stream)
    for k in range(K):
        for n in names:
            a, b = ev[n][k]
            a.record(stream)
            call(n, inputs[n]["x"], outputs[n])
            b.record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks.stop()
    barrier()
    secs = t_start.elapsed_time(t_end) / 1e3
    step_bytes = sum(alg_bytes(wl) for wl in wls.values())
    secs_max, total_bytes = aggregate(secs, step_bytes * K)
    per_op = {}
    for n in names:
        ms = [a.elapsed_time(b) for a, b in ev[n]]
        avg_s = statistics.fmean(ms) / 1e3
        per_op[n] = {"avg_ms": avg_s * 1e3, "median_ms": statistics.median(ms), "min_ms": min(ms),
                     "gbs": alg_bytes(wls[n]) / avg_s / 1e9, "rows_per_s": wls[n].M / avg_s}
    peak, peak_kind = measured_peak()
    for n in names:
        fr = fractions(per_op[n]["gbs"], peak, copy_gbs)
        per_op[n]["frac_of_" + peak_kind] = fr["frac"]
        per_op[n]["frac_of_in_run_copy"] = fr["frac_of_in_run_copy"]
        per_op[n]["frac_of_nominal"] = fr["frac_of_nominal"]
    # kernels of one step, counted from the CUDA activity trace after the timed region
    per_step = count_kernels(lambda: [call(n, inputs[n]["x"], outputs[n]) for n in names])
    launches_from = "cuda activity trace of one step"
    if per_step is None:
        per_step = sum(KERNELS_PER_CALL[wls[n].op] for n in names)
        launches_from = "per-operation table"
    launches = K * per_step

    # end to end through the public API, host buffers: H2D inputs, kernels, D2H outputs
    e2e = None
    if not args.no_e2e:
        host_in = {n: inputs[n]["x"].cpu().pin_memory() for n in names}
        result = {n: reds.get(n, outputs[n]) for n in names}  # what each call produces
        host_out = {n: torch.empty(result[n].shape, dtype=result[n].dtype).pin_memory() for n in names}
        host_wb = {n: {k: inputs[n][k].cpu().pin_memory() for k in ("w", "b", "residual", "dy") if k in inputs[n]}
                   for n in names}
        host_ro = {n: torch.empty(res_out[n].shape, dtype=res_out[n].dtype).pin_memory() for n in res_out}
        h2d = sum(t.numel() * t.element_size() for t in host_in.values()) + \
            sum(t.numel() * t.element_size() for d in host_wb.values() for t in d.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out.values()) + \
            sum(t.numel() * t.element_size() for t in host_ro.values())
        ke = max(2, min(K, args.e2e_steps))
        # three streams: host->device copies, the library calls, device->host
        # copies (separate copy engines, so the two directions overlap). Per
        # workload, a step's input copies wait until the previous step's call
        # has read its inputs, and its call until the previous step's result
        # has been copied out.
        s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        called = {n: None for n in names}
        drained = {n: None for n in names}

        def e2e_step(calls=True):
            for n in names:
                with torch.cuda.stream(s_in):
                    if called[n] is not None:
                        s_in.wait_event(called[n])
                    for kk, t in host_wb[n].items():
                        inputs[n][kk].copy_(t, non_blocking=True)
                    inputs[n]["x"].copy_(host_in[n], non_blocking=True)
                    loaded = torch.cuda.Event()
                    loaded.record(s_in)
                with torch.cuda.stream(s_run):
                    s_run.wait_event(loaded)
                    if drained[n] is not None:
                        s_run.wait_event(drained[n])
                    if calls:
                        call(n, inputs[n]["x"], outputs[n])
                    called[n] = torch.cuda.Event()
                    called[n].record(s_run)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(called[n])
                    host_out[n].copy_(result[n], non_blocking=True)
                    if n in host_ro:
                        host_ro[n].copy_(res_out[n], non_blocking=True)
                    drained[n] = torch.cuda.Event()
                    drained[n].record(s_out)

        def timed(calls):
            e2e_step(calls)
            torch.cuda.synchronize()
            barrier()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s_in)
            for _ in range(ke):
                e2e_step(calls)
            s_in.wait_stream(s_run)
            s_in.wait_stream(s_out)
            b.record(s_in)
            torch.cuda.synchronize()
            barrier()
            return a.elapsed_time(b) / 1e3

        es, eb = aggregate(timed(True), step_bytes * ke)
        # the host link's ceiling in the same run: the same three-stream
        # pipeline with every copy and no kernel
        cs, _ = aggregate(timed(False), 0.0)
        ceiling = link_ceiling(step_bytes, cs, ke)
        e2e = {"value": eb / es / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": ke, "ms_per_step": es / ke * 1e3,
               "host_link": {"copies_only_ms_per_step": cs / ke * 1e3,
                             "h2d_plus_d2h_gbs": (h2d + d2h) * ke / cs / 1e9,
                             "ceiling": ceiling, "frac_of_ceiling": (eb / es / 1e9) / ceiling}}

    extras = None
    if rank == 0 and not args.no_extras and not subset and args.rows_scale == 1.0:
        extras = run_extras(dev, stream)

    eager = None
    if rank == 0 and not args.no_torch_eager and not subset and args.rows_scale == 1.0:
        eager = run_torch_eager(wls, inputs, stream)

    host_cost = None
    if rank == 0 and not args.no_extras and not subset and args.rows_scale == 1.0:
        host_cost = {"python_us_per_call": host_cost_python(dev), "c": host_cost_c(),
                     "what": "rowops_softmax on fp32 1024 x 768: host time to issue one call (Python binding; "
                             "C driver tests/native/host_cost.c with its event and CUDA-graph figures)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import oracle

        oracle.build()
        threads = host_threads()
        v, sample, spent = cpu_baseline(oracle, dev_inputs=inputs, budget_s=args.cpu_budget_s / 2, threads=threads,
                                        wls=wls)
        v1, sample1, spent1 = cpu_baseline(oracle, dev_inputs=inputs, budget_s=args.cpu_budget_s / 2, threads=1,
                                           wls=wls)
        cpu = {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample,
               "seconds": spent, "single_core": {"value": v1, "sample": sample1, "seconds": spent1}}

    if rank != 0:
        return 0
    roof = None
    if DOMINANT in per_op:
        ach = per_op[DOMINANT]["gbs"]
        fr = fractions(ach, peak, copy_gbs)
        roof = {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": fr["frac"],
                "peak_kind": peak_kind,
                "in_run_copy": {"gbs": copy_gbs, "frac": fr["frac_of_in_run_copy"],
                                "how": "cudaMemcpyAsync device to device of 1 GiB, read + write bytes, best of 10"},
                "nominal": {"gbs": NOMINAL_HBM_GBS, "frac": fr["frac_of_nominal"]}, "kernel": "ln_gelu_tma_kernel<bf16, 128 threads/row, 8 vectors/thread, 5 rows/CTA, full rows>",
                "traffic": profiled_traffic() if args.rows_scale == 1.0 else None,
                "algorithmic_bytes_per_launch": alg_bytes(wls[DOMINANT])}
    line = {
        "metric": METRIC,
        "value": total_bytes / secs_max / 1e9,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": secs_max / K * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": STEP_DTYPE if not subset else "f32 arithmetic; I/O " + ", ".join(
            sorted({wl.dtype for wl in wls.values()})),
        "data": "synthetic",
        "config": config_block(world) if args.rows_scale == 1.0 and not subset else
        {"workload": " + ".join(f"{wl.name}[M={wl.M}]" for wl in wls.values()), "parallelism": parallelism(world)},
        "roofline": roof,
        "step_frac": fractions(total_bytes / secs_max / 1e9, peak, copy_gbs),
        "breakdown": per_op,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "gpu_launches_from": launches_from,
        "extras": extras,
        "host_cost": host_cost,
        "context_torch_eager": eager,
        "clocks": clocks.summary(),
        "device": torch.cuda.get_device_name(dev),
        "num_sms": torch.cuda.get_device_properties(dev).multi_processor_count,
    }
    print(json.dumps(line))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["rowops", "reference"], default="rowops")
    ap.add_argument("--ops", default="", help="comma-separated subset of softmax,online,layernorm (profiling)")
    ap.add_argument("--rows-scale", type=float, default=1.0, help="scale every workload's rows (profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the small and ragged-tail workloads")
    ap.add_argument("--no-torch-eager", action="store_true", help="skip the PyTorch eager context timings")
    ap.add_argument("--workloads", default="",
                    help="comma-separated workload names to time as the step instead of the default (profiling)")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--reference-budget-s", type=float, default=90.0)
    ap.add_argument("--clocks-csv", default=None, help="also log nvidia-smi clock samples to this CSV")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "rowops":
        args.warmup = 3
    return run_reference(args) if args.impl == "reference" else run_rowops(args)


if __name__ == "__main__":
    sys.exit(main())
