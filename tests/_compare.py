"""Element-wise comparison of CUDA results with the oracle, with the
tolerances the specification states:

* fp32 softmax (plain and online): max relative error 1e-5;
* fp32 LayerNorm+GELU: max absolute error 1e-5;
* bf16 output: within 1 bf16 ulp of the oracle's double value (fp32
  accumulation inside, round to nearest even on the way out).

Two floors come from fp32 arithmetic itself, and each is stated where used:
exponentials below the smallest normal fp32 (2^-126) are flushed to zero, so
softmax allows an absolute 2^-126; and LayerNorm+GELU in bf16 allows the fp32
path's own absolute 1e-5 on top of the ulp, because near a zero of the affine
output z the fp32 rounding of the statistics is larger than one bf16 ulp of
the tiny result.
"""
from __future__ import annotations

import numpy as np
import torch

FTZ_FLOOR = 2.0 ** -126


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of an fp32 / bf16 tensor to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float32).numpy().astype(np.float64)


def to_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float32).numpy()


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """One bf16 ulp at |v| (8 significant bits); the subnormal spacing below 2^-126."""
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, FTZ_FLOOR)))
    return np.exp2(e - 7.0)


def _check_nan(got, ref, what):
    rn = np.isnan(ref)
    gn = np.isnan(got)
    bad = rn != gn
    assert not bad.any(), f"{what}: NaN mismatch at {np.argwhere(bad)[:5].tolist()}"
    return ~rn


def assert_softmax_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "softmax"):
    got = np.asarray(got, dtype=np.float64)
    ok = _check_nan(got, ref, what)
    g, r = got[ok], ref[ok]
    zero = r == 0.0
    assert np.all(g[zero] == 0.0), f"{what}: masked entries must be exactly 0"
    if dtype == "f32":
        tol = 1e-5 * np.abs(r) + FTZ_FLOOR
    else:
        tol = bf16_ulp(r) + FTZ_FLOOR
    err = np.abs(g - r)
    worst = np.argmax(err - tol) if err.size else 0
    assert np.all(err <= tol), (
        f"{what}: max excess {float((err - tol).max()):.3e} at got={g.flat[worst]!r} ref={r.flat[worst]!r}"
    )
    return float((err / np.maximum(np.abs(r), FTZ_FLOOR)).max()) if err.size else 0.0


def assert_ln_gelu_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "layernorm_gelu",
                         rel: float = 0.0):
    """``rel`` adds a relative allowance for edge cases whose outputs are far
    larger than the workloads' (an fp32 ulp at |z| = 300 is 3e-5 on its own)."""
    got = np.asarray(got, dtype=np.float64)
    ok = _check_nan(got, ref, what)
    g, r = got[ok], ref[ok]
    if dtype == "f32":
        tol = np.full_like(r, 1e-5)
    else:
        tol = bf16_ulp(r) + 1e-5
    tol = tol + rel * np.abs(r)
    err = np.abs(g - r)
    worst = np.argmax(err - tol) if err.size else 0
    assert np.all(err <= tol), (
        f"{what}: max excess {float((err - tol).max()):.3e} at got={g.flat[worst]!r} ref={r.flat[worst]!r}"
    )
    return float(err.max()) if err.size else 0.0


def assert_rms_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "rmsnorm", rel: float = 0.0):
    """RMSNorm outputs: fp32 max absolute error 1e-5 (the fp32 bar of the
    LayerNorm+GELU workloads, whose outputs have the same O(1) magnitude);
    bf16 within 1 bf16 ulp. y = s * inv_rms * w has no cancellation, so no
    extra floor. ``rel`` as for assert_ln_gelu_close."""
    got = np.asarray(got, dtype=np.float64)
    ok = _check_nan(got, ref, what)
    g, r = got[ok], ref[ok]
    tol = np.full_like(r, 1e-5) if dtype == "f32" else bf16_ulp(r)
    tol = tol + rel * np.abs(r)
    err = np.abs(g - r)
    worst = np.argmax(err - tol) if err.size else 0
    assert np.all(err <= tol), (
        f"{what}: max excess {float((err - tol).max()):.3e} at got={g.flat[worst]!r} ref={r.flat[worst]!r}"
    )
    return float(err.max()) if err.size else 0.0
