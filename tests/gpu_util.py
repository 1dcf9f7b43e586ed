"""Helpers for the GPU parity tests: device set-up, strided buffers with guard
bands, and oracle evaluation of sampled rows."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from row_wise_reduction_gb300 import workloads

requires_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")

SENTINEL_F32 = 3072.0  # exact in fp32 and bf16; no softmax or GELU output of these tests equals it


def dev():
    return torch.device("cuda", torch.cuda.current_device())


def make_x(wl: workloads.Workload, ld=None, offset=0, device=None):
    """Inputs of ``wl`` on the GPU; x is an (M, N) view into storage of row
    stride ``ld`` starting ``offset`` elements in (so rows can be misaligned)."""
    device = device or dev()
    ld = wl.N if ld is None else ld
    inp = workloads.make_inputs(wl, device=device, ld=ld)
    if offset:
        st = torch.full((wl.M * ld + offset + 8,), float("nan"), dtype=inp["x"].dtype, device=device)
        view = st[offset:offset + wl.M * ld].view(wl.M, ld)
        view.copy_(inp["x_storage"])
        inp["x_storage"] = view
        inp["x"] = view[:, : wl.N]
        inp["base"] = st
    return inp


def guarded_like(x: torch.Tensor, offset: int = 0, guard: int = 64):
    """An output view shaped and strided like ``x`` inside a buffer whose every
    element outside the view holds a sentinel. Returns (view, buffer, mask of
    the view's elements within the buffer)."""
    M, N = x.shape
    ld = x.stride(0) if M > 1 else N
    total = guard + offset + (M - 1) * ld + N + guard
    buf = torch.full((total,), SENTINEL_F32, dtype=x.dtype, device=x.device)
    start = guard + offset
    view = torch.as_strided(buf, (M, N), (ld, 1), start)
    inside = torch.zeros(total, dtype=torch.bool)
    idx = start + (torch.arange(M).unsqueeze(1) * ld + torch.arange(N).unsqueeze(0))
    inside[idx.reshape(-1)] = True
    return view, buf, inside


def assert_guard_untouched(buf: torch.Tensor, inside: torch.Tensor):
    b = buf.detach().float().cpu()
    out = b[~inside]
    assert torch.all(out == SENTINEL_F32), "a kernel wrote outside its rows"


def rows_f32(t: torch.Tensor, rows=None) -> np.ndarray:
    """fp32 numpy copy of (sampled) rows of a CUDA tensor; bf16 widens exactly."""
    if rows is not None:
        t = t[torch.as_tensor(rows, device=t.device)]
    return t.detach().float().cpu().numpy()


def sample_rows(M: int, k: int, seed: int = 0):
    """First, last and k - 2 seeded random rows."""
    if M <= k:
        return list(range(M))
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, M - 1), size=k - 2, replace=False)
    return sorted({0, M - 1, *mid.tolist()})
