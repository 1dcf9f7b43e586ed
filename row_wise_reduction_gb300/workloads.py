"""Seeded synthetic inputs for the row-wise reduce-then-normalise workloads.

This module holds random-number generation and the workload table (shapes,
dtypes, value distributions, masking and outlier structure) and nothing of the
operations' arithmetic. The CUDA path's tests and benchmark and the oracle's
tests all draw their inputs from here, so both sides see identical values.

Inputs are drawn with a ``torch.Generator`` on the requested device, seeded per
workload: values generated on the CPU and on a GPU follow the same recipe but
are different streams. Large workloads are generated on the device (CPU
generation of the 1 GiB case takes most of a minute) and the rows the oracle
checks are copied back to the host.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "torch_dtype", "elem_size"]


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: an operation, a dtype, a shape and a value recipe."""

    name: str
    op: str  # "softmax" | "softmax_causal" | "online_softmax" | "layernorm_gelu" | "layernorm_gelu_erf" |
    #          "layernorm_gelu_backward" | "rmsnorm" | "residual_rmsnorm" | "row_sum" | "row_max" |
    #          "bias_residual_gelu"
    dtype: str  # "f32" | "bf16"
    M: int  # rows
    N: int  # columns (reduction length)
    seed: int  # seed of x; w, b, the residual and dy use seed + 100, + 200, + 300 and + 400
    x_std: float = 1.0  # x ~ N(0, x_std^2)
    causal: bool = False  # row r keeps columns c <= r mod N, the rest are -inf
    outlier_p: float = 0.0  # fraction of entries (Bernoulli per entry) set to outlier_value
    outlier_value: float = 30.0
    affine: bool = False  # w ~ U(0.5, 1.5), b ~ N(0, 0.1^2) (RMSNorm uses w only)
    residual: bool = False  # a second input of the same shape, ~ N(0, 1)
    grad: bool = False  # an upstream gradient dy of the same shape, ~ N(0, 1)
    eps: float = 1e-5

    def with_shape(self, M: Optional[int] = None, N: Optional[int] = None) -> "Workload":
        return dataclasses.replace(self, M=self.M if M is None else M, N=self.N if N is None else N)


# The benchmark workloads of softmax, split-row softmax and LayerNorm+GELU (with
# the two ragged-tail variants of the bf16 LayerNorm+GELU case) and of RMSNorm,
# keyed by a descriptive name.
WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("softmax_f32_1024x768", "softmax", "f32", 1024, 768, seed=0),
        Workload("layernorm_gelu_f32_4096x768", "layernorm_gelu", "f32", 4096, 768, seed=1, affine=True),
        Workload("softmax_bf16_causal_32768x4096", "softmax", "bf16", 32768, 4096, seed=2, x_std=2.0, causal=True),
        Workload("online_softmax_f32_64x1048576", "online_softmax", "f32", 64, 1 << 20, seed=3, outlier_p=1e-3),
        Workload("layernorm_gelu_bf16_65536x8192", "layernorm_gelu", "bf16", 65536, 8192, seed=4, affine=True),
        Workload("layernorm_gelu_bf16_65536x127", "layernorm_gelu", "bf16", 65536, 127, seed=4, affine=True),
        Workload("layernorm_gelu_bf16_65536x4097", "layernorm_gelu", "bf16", 65536, 4097, seed=4, affine=True),
        # the causal softmax entry point on the causal softmax input (period N, offset 0: row r keeps
        # columns c <= r mod N) [Triton Kernel 实现练习 §5.1]
        Workload("softmax_causal_bf16_32768x4096", "softmax_causal", "bf16", 32768, 4096, seed=2, x_std=2.0,
                 causal=True),
        # RMSNorm and fused residual + RMSNorm [Triton Kernel 实现练习 §4.2, §4.3], on the shapes of
        # the LayerNorm+GELU workloads
        Workload("rmsnorm_f32_4096x768", "rmsnorm", "f32", 4096, 768, seed=5, affine=True),
        Workload("rmsnorm_bf16_65536x8192", "rmsnorm", "bf16", 65536, 8192, seed=6, affine=True),
        Workload("residual_rmsnorm_f32_4096x768", "residual_rmsnorm", "f32", 4096, 768, seed=7, affine=True,
                 residual=True),
        Workload("residual_rmsnorm_bf16_65536x8192", "residual_rmsnorm", "bf16", 65536, 8192, seed=8, affine=True,
                 residual=True),
        # LayerNorm + exact (erf) GELU [Triton Kernel 实现练习 §3.4] on the LayerNorm+GELU inputs, and
        # the row-wise sum / max [§2.2, §2.3] on the shape of the large LayerNorm+GELU input
        Workload("layernorm_gelu_erf_f32_4096x768", "layernorm_gelu_erf", "f32", 4096, 768, seed=1, affine=True),
        Workload("layernorm_gelu_erf_bf16_65536x8192", "layernorm_gelu_erf", "bf16", 65536, 8192, seed=4,
                 affine=True),
        Workload("row_sum_bf16_65536x8192", "row_sum", "bf16", 65536, 8192, seed=9),
        Workload("row_max_bf16_65536x8192", "row_max", "bf16", 65536, 8192, seed=10),
        # the backward of LayerNorm -> affine -> tanh-GELU [PyTorch 自定义 CUDA 算子与 Triton 编程
        # §三 FusedLayerNormGELU] on the LayerNorm+GELU inputs, with dy ~ N(0, 1)
        Workload("layernorm_gelu_backward_f32_4096x768", "layernorm_gelu_backward", "f32", 4096, 768, seed=1,
                 affine=True, grad=True),
        Workload("layernorm_gelu_backward_bf16_65536x8192", "layernorm_gelu_backward", "bf16", 65536, 8192,
                 seed=4, affine=True, grad=True),
        # fused residual + bias + GELU [Triton Kernel 实现练习 §3.4] on the LayerNorm+GELU shapes: x,
        # residual ~ N(0, 1), the bias is the affine b ~ N(0, 0.1^2)
        Workload("bias_residual_gelu_f32_4096x768", "bias_residual_gelu", "f32", 4096, 768, seed=11, affine=True,
                 residual=True),
        Workload("bias_residual_gelu_bf16_65536x8192", "bias_residual_gelu", "bf16", 65536, 8192, seed=12,
                 affine=True, residual=True),
    ]
}


def torch_dtype(dtype: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


def elem_size(dtype: str) -> int:
    return {"f32": 4, "bf16": 2}[dtype]


def _gen(device: torch.device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_inputs(
    wl: Workload,
    device: str | torch.device = "cpu",
    ld: Optional[int] = None,
    row_ids: Optional[torch.Tensor] = None,
    block: int = 0,
) -> Dict[str, torch.Tensor]:
    """Draw the inputs of ``wl`` on ``device``.

    Returns ``{"x": (M, N) view, "x_storage": (M, ld) tensor}``, for affine
    workloads ``"w"`` and ``"b"`` of length N, and for residual workloads
    ``"residual"`` / ``"residual_storage"`` laid out like x, for gradient
    workloads ``"dy"`` / ``"dy_storage"`` likewise. Values are drawn in
    fp32 and rounded to the workload's dtype (round to nearest even). With
    ``ld > N`` the padding columns of each row hold NaN so that any read past
    column N-1 shows up in the result. ``row_ids`` (M integers) gives the row
    index each generated row stands for in the causal mask pattern, so that a
    small sample can carry the mask of rows spread over a large workload.
    ``block`` b > 0: rows [b M, (b + 1) M) of a larger problem made of such
    blocks (one per rank of a multi-GPU run): its own draw (seed + 7919 b) and,
    for causal workloads, the mask of those global row indices; w and b are
    the problem's, shared by every block.
    """
    device = torch.device(device)
    M, N = wl.M, wl.N
    ld = N if ld is None else ld
    if ld < N:
        raise ValueError("ld must be >= N")
    dt = torch_dtype(wl.dtype)
    g = _gen(device, wl.seed + 7919 * block)
    x = torch.randn((M, N), generator=g, device=device, dtype=torch.float32)
    if wl.x_std != 1.0:
        x.mul_(wl.x_std)
    if wl.outlier_p > 0.0:
        hit = torch.rand((M, N), generator=g, device=device, dtype=torch.float32) < wl.outlier_p
        x.masked_fill_(hit, wl.outlier_value)
        del hit
    if wl.causal:
        cols = torch.arange(N, device=device).unsqueeze(0)
        ids = (torch.arange(M, device=device) + int(block) * M if row_ids is None
               else torch.as_tensor(row_ids, device=device))
        keep = (ids % N).unsqueeze(1)
        x.masked_fill_(cols > keep, float("-inf"))
    storage = torch.full((M, ld), float("nan"), device=device, dtype=dt)
    storage[:, :N] = x.to(dt)
    del x
    out = {"x": storage[:, :N], "x_storage": storage}
    if wl.affine:
        gw = _gen(device, wl.seed + 100)
        gb = _gen(device, wl.seed + 200)
        w = 0.5 + torch.rand((N,), generator=gw, device=device, dtype=torch.float32)
        b = 0.1 * torch.randn((N,), generator=gb, device=device, dtype=torch.float32)
        out["w"] = w.to(dt)
        out["b"] = b.to(dt)
    for key, on, sd in (("residual", wl.residual, 300), ("dy", wl.grad, 400)):
        if on:
            gr = _gen(device, wl.seed + sd + 7919 * block)
            r = torch.randn((M, N), generator=gr, device=device, dtype=torch.float32)
            rs = torch.full((M, ld), float("nan"), device=device, dtype=dt)
            rs[:, :N] = r.to(dt)
            del r
            out[key] = rs[:, :N]
            out[key + "_storage"] = rs
    return out
