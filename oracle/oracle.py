"""Python access to the double-precision CPU oracle (``rowops_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the test suite, by the package smoke
check and by the benchmark's CPU-baseline leg. The product path never imports
it. Arrays go in as numpy (float32 values, which hold bf16 values exactly, or
float64 for the single-row forms) and come out as float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rowops_oracle.c")
_LIB = os.path.join(_HERE, "librowops_oracle.so")

_c_double_p = ctypes.POINTER(ctypes.c_double)
_c_float_p = ctypes.POINTER(ctypes.c_float)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with the system C compiler (IEEE double, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "rowops_oracle.h"))
    ):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.oracle_gelu_sqrt_2_over_pi.restype = ctypes.c_double
        L.oracle_gelu_cubic.restype = ctypes.c_double
        L.oracle_gelu_tanh.restype = ctypes.c_double
        L.oracle_gelu_tanh.argtypes = [ctypes.c_double]
        L.oracle_softmax_row.argtypes = [_c_double_p, _i64, _c_double_p]
        L.oracle_online_softmax_row.argtypes = [_c_double_p, _i64, _i64, _c_double_p, _c_double_p, _c_double_p]
        L.oracle_split_softmax_row.argtypes = [_c_double_p, _i64, _i64, _c_double_p, _c_double_p, _c_double_p]
        L.oracle_layernorm_row.argtypes = [_c_double_p, _c_double_p, _c_double_p, ctypes.c_double, _i64, _c_double_p]
        L.oracle_layernorm_gelu_row.argtypes = L.oracle_layernorm_row.argtypes
        for name in ("oracle_softmax_rows_f32",):
            getattr(L, name).argtypes = [_c_float_p, _i64, _i64, _i64, _c_double_p]
            getattr(L, name).restype = ctypes.c_int
        L.oracle_split_softmax_rows_f32.argtypes = [_c_float_p, _i64, _i64, _i64, _i64, _c_double_p]
        L.oracle_split_softmax_rows_f32.restype = ctypes.c_int
        for name in ("oracle_layernorm_gelu_rows_f32", "oracle_layernorm_rows_f32"):
            getattr(L, name).argtypes = [_c_float_p, _c_float_p, _c_float_p, ctypes.c_double, _i64, _i64, _i64,
                                         _c_double_p]
            getattr(L, name).restype = ctypes.c_int
        L.oracle_rmsnorm_row.argtypes = [_c_double_p, _c_double_p, ctypes.c_double, _i64, _c_double_p]
        L.oracle_gelu_tanh_grad.argtypes = [ctypes.c_double]
        L.oracle_gelu_tanh_grad.restype = ctypes.c_double
        L.oracle_layernorm_gelu_backward_row.argtypes = [_c_double_p, _c_double_p, _c_double_p, _c_double_p,
                                                         ctypes.c_double, _i64, _c_double_p, _c_double_p, _c_double_p]
        L.oracle_layernorm_gelu_backward_rows_f32.argtypes = [_c_float_p, _c_float_p, _c_float_p, _c_float_p,
                                                              ctypes.c_double, _i64, _i64, _i64, _c_double_p,
                                                              _c_double_p, _c_double_p]
        L.oracle_layernorm_gelu_backward_rows_f32.restype = ctypes.c_int
        L.oracle_gelu_erf.argtypes = [ctypes.c_double]
        L.oracle_gelu_erf.restype = ctypes.c_double
        L.oracle_layernorm_gelu_erf_rows_f32.argtypes = [_c_float_p, _c_float_p, _c_float_p, ctypes.c_double, _i64,
                                                         _i64, _i64, _c_double_p]
        L.oracle_layernorm_gelu_erf_rows_f32.restype = ctypes.c_int
        for name in ("oracle_row_sum_rows_f32", "oracle_row_max_rows_f32"):
            getattr(L, name).argtypes = [_c_float_p, _i64, _i64, _i64, _c_double_p]
            getattr(L, name).restype = ctypes.c_int
        L.oracle_causal_kept.argtypes = [_i64, _i64, _i64, _i64]
        L.oracle_causal_kept.restype = _i64
        L.oracle_softmax_causal_rows_f32.argtypes = [_c_float_p, _i64, _i64, _i64, _i64, _i64, _c_double_p]
        L.oracle_softmax_causal_rows_f32.restype = ctypes.c_int
        L.oracle_round_to.argtypes = [ctypes.c_double, ctypes.c_int]
        L.oracle_round_to.restype = ctypes.c_double
        L.oracle_residual_rmsnorm_row.argtypes = [_c_double_p, _c_double_p, _c_double_p, ctypes.c_double, _i64,
                                                  ctypes.c_int, _c_double_p, _c_double_p]
        L.oracle_rmsnorm_rows_f32.argtypes = [_c_float_p, _c_float_p, ctypes.c_double, _i64, _i64, _i64,
                                              _c_double_p]
        L.oracle_rmsnorm_rows_f32.restype = ctypes.c_int
        L.oracle_residual_rmsnorm_rows_f32.argtypes = [_c_float_p, _c_float_p, _c_float_p, ctypes.c_double,
                                                       ctypes.c_int, _i64, _i64, _i64, _c_double_p, _c_double_p]
        L.oracle_residual_rmsnorm_rows_f32.restype = ctypes.c_int
        L.oracle_bias_residual_gelu_rows_f32.argtypes = [_c_float_p, _c_float_p, _c_float_p, _i64, _i64, _i64,
                                                          ctypes.c_int, _c_double_p]
        L.oracle_bias_residual_gelu_rows_f32.restype = ctypes.c_int
        _lib = L
    return _lib


def _dp(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(_c_double_p)


def _fp(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(_c_float_p)


def _rows(x: np.ndarray) -> Tuple[np.ndarray, int, int, int]:
    """Return a float32 2-D array with unit column stride, plus (M, N, ld)."""
    x = np.asarray(x)
    if x.ndim == 1:
        x = x[None, :]
    if x.ndim != 2:
        raise ValueError("expected a 1-D or 2-D array")
    if x.dtype != np.float32 or x.strides[1] != 4 or x.strides[0] % 4 != 0 or x.strides[0] < 4 * x.shape[1]:
        x = np.ascontiguousarray(x, dtype=np.float32)
    M, N = x.shape
    ld = x.strides[0] // 4 if M > 1 else N
    return x, M, N, ld


def _f64_row(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64).reshape(-1))


def _opt32(v, N) -> Optional[np.ndarray]:
    if v is None:
        return None
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32).reshape(-1))
    if v.shape[0] != N:
        raise ValueError("w / b must have N entries")
    return v


def _opt64(v, N) -> Optional[np.ndarray]:
    if v is None:
        return None
    v = _f64_row(v)
    if v.shape[0] != N:
        raise ValueError("w / b must have N entries")
    return v


# ---- constants ---------------------------------------------------------------
def gelu_sqrt_2_over_pi() -> float:
    return lib().oracle_gelu_sqrt_2_over_pi()


def gelu_cubic() -> float:
    return lib().oracle_gelu_cubic()


# ---- single rows in double -----------------------------------------------------
def softmax_row(x) -> np.ndarray:
    xr = _f64_row(x)
    y = np.empty_like(xr)
    lib().oracle_softmax_row(_dp(xr), xr.size, _dp(y))
    return y


def online_softmax_row(x, block: int) -> Tuple[np.ndarray, float, float]:
    xr = _f64_row(x)
    y = np.empty_like(xr)
    m = ctypes.c_double()
    d = ctypes.c_double()
    lib().oracle_online_softmax_row(_dp(xr), xr.size, int(block), _dp(y), ctypes.byref(m), ctypes.byref(d))
    return y, m.value, d.value


def split_softmax_row(x, chunk: int) -> Tuple[np.ndarray, float, float]:
    xr = _f64_row(x)
    y = np.empty_like(xr)
    m = ctypes.c_double()
    d = ctypes.c_double()
    lib().oracle_split_softmax_row(_dp(xr), xr.size, int(chunk), _dp(y), ctypes.byref(m), ctypes.byref(d))
    return y, m.value, d.value


def layernorm_row(x, w=None, b=None, eps: float = 1e-5) -> np.ndarray:
    xr = _f64_row(x)
    z = np.empty_like(xr)
    wd, bd = _opt64(w, xr.size), _opt64(b, xr.size)
    lib().oracle_layernorm_row(_dp(xr), _dp(wd), _dp(bd), float(eps), xr.size, _dp(z))
    return z


def layernorm_gelu_row(x, w=None, b=None, eps: float = 1e-5) -> np.ndarray:
    xr = _f64_row(x)
    y = np.empty_like(xr)
    wd, bd = _opt64(w, xr.size), _opt64(b, xr.size)
    lib().oracle_layernorm_gelu_row(_dp(xr), _dp(wd), _dp(bd), float(eps), xr.size, _dp(y))
    return y


STORAGE = {"exact": 0, "f32": 1, "bf16": 2}


def round_to(v, storage: str) -> np.ndarray:
    """Round to nearest even in the storage type ("exact", "f32", "bf16")."""
    f = lib().oracle_round_to
    code = STORAGE[storage]
    vv = np.asarray(v, dtype=np.float64)
    return np.vectorize(lambda t: f(t, code), otypes=[np.float64])(vv) if vv.ndim else np.float64(f(float(vv), code))


def rmsnorm_row(x, w=None, eps: float = 1e-5) -> np.ndarray:
    xr = _f64_row(x)
    y = np.empty_like(xr)
    lib().oracle_rmsnorm_row(_dp(xr), _dp(_opt64(w, xr.size)), float(eps), xr.size, _dp(y))
    return y


def residual_rmsnorm_row(x, r, w=None, eps: float = 1e-5, storage: str = "exact") -> Tuple[np.ndarray, np.ndarray]:
    """(residual_out, out) of one row."""
    xr, rr = _f64_row(x), _f64_row(r)
    if rr.size != xr.size:
        raise ValueError("x and residual must have the same length")
    s_out, y = np.empty_like(xr), np.empty_like(xr)
    lib().oracle_residual_rmsnorm_row(_dp(xr), _dp(rr), _dp(_opt64(w, xr.size)), float(eps), xr.size,
                                      STORAGE[storage], _dp(s_out), _dp(y))
    return s_out, y


def gelu_tanh(z) -> np.ndarray:
    f = lib().oracle_gelu_tanh
    zz = np.asarray(z, dtype=np.float64)
    return np.vectorize(f, otypes=[np.float64])(zz) if zz.ndim else np.float64(f(float(zz)))


# ---- row batches (fp32-valued inputs) --------------------------------------------
def softmax(x) -> np.ndarray:
    """Stable softmax of every row of a 2-D fp32-valued array -> float64 (M, N)."""
    xs, M, N, ld = _rows(x)
    y = np.empty((M, N), dtype=np.float64)
    if lib().oracle_softmax_rows_f32(_fp(xs), M, N, ld, _dp(y)) != 0:
        raise ValueError("oracle_softmax_rows_f32 rejected its arguments")
    return y


def split_softmax(x, chunk: int) -> np.ndarray:
    """Split-row softmax (chunk partials merged in a second pass) -> float64 (M, N)."""
    xs, M, N, ld = _rows(x)
    y = np.empty((M, N), dtype=np.float64)
    if lib().oracle_split_softmax_rows_f32(_fp(xs), M, N, ld, int(chunk), _dp(y)) != 0:
        raise ValueError("oracle_split_softmax_rows_f32 rejected its arguments")
    return y


def layernorm_gelu(x, w=None, b=None, eps: float = 1e-5) -> np.ndarray:
    """LayerNorm -> affine -> tanh-GELU of every row -> float64 (M, N)."""
    xs, M, N, ld = _rows(x)
    y = np.empty((M, N), dtype=np.float64)
    wf, bf = _opt32(w, N), _opt32(b, N)
    if lib().oracle_layernorm_gelu_rows_f32(_fp(xs), _fp(wf), _fp(bf), float(eps), M, N, ld, _dp(y)) != 0:
        raise ValueError("oracle_layernorm_gelu_rows_f32 rejected its arguments")
    return y


def layernorm(x, w=None, b=None, eps: float = 1e-5) -> np.ndarray:
    """LayerNorm -> affine (no GELU) of every row -> float64 (M, N)."""
    xs, M, N, ld = _rows(x)
    y = np.empty((M, N), dtype=np.float64)
    wf, bf = _opt32(w, N), _opt32(b, N)
    if lib().oracle_layernorm_rows_f32(_fp(xs), _fp(wf), _fp(bf), float(eps), M, N, ld, _dp(y)) != 0:
        raise ValueError("oracle_layernorm_rows_f32 rejected its arguments")
    return y


def rmsnorm(x, w=None, eps: float = 1e-5) -> np.ndarray:
    """RMSNorm of every row -> float64 (M, N)."""
    xs, M, N, ld = _rows(x)
    y = np.empty((M, N), dtype=np.float64)
    if lib().oracle_rmsnorm_rows_f32(_fp(xs), _fp(_opt32(w, N)), float(eps), M, N, ld, _dp(y)) != 0:
        raise ValueError("oracle_rmsnorm_rows_f32 rejected its arguments")
    return y


def residual_rmsnorm(x, r, w=None, eps: float = 1e-5, storage: str = "exact") -> Tuple[np.ndarray, np.ndarray]:
    """Fused residual + RMSNorm of every row -> (residual_out, out), float64 (M, N) each;
    residual_out rounded to `storage` ("exact", "f32", "bf16") before the norm."""
    xs, M, N, ld = _rows(x)
    rs, Mr, Nr, ldr = _rows(r)
    if (Mr, Nr) != (M, N):
        raise ValueError("x and residual must have the same shape")
    if ldr != ld:  # the batch form takes one row stride for both
        xs, rs, ld = np.ascontiguousarray(xs), np.ascontiguousarray(rs), N
    s_out = np.empty((M, N), dtype=np.float64)
    y = np.empty((M, N), dtype=np.float64)
    if lib().oracle_residual_rmsnorm_rows_f32(_fp(xs), _fp(rs), _fp(_opt32(w, N)), float(eps), STORAGE[storage],
                                              M, N, ld, _dp(s_out), _dp(y)) != 0:
        raise ValueError("oracle_residual_rmsnorm_rows_f32 rejected its arguments")
    return s_out, y


def causal_kept(r: int, n: int, period: int, offset: int = 0) -> int:
    """Columns of row r kept by the causal mask (c <= r mod period + offset)."""
    return int(lib().oracle_causal_kept(int(r), int(n), int(period), int(offset)))


def softmax_causal(x, period: int, offset: int = 0, row0: int = 0) -> np.ndarray:
    """Causal softmax of every row -> float64 (M, N). ``row0``: index of the
    first given row in the full matrix (for sampled rows, contiguous from row0)."""
    xs, M, N, ld = _rows(x)
    y = np.empty((M, N), dtype=np.float64)
    if row0:
        # the mask depends on the row index: evaluate row by row at its own index
        for i in range(M):
            y[i] = softmax_causal_rows_at(xs[i], row0 + i, period, offset)
        return y
    if lib().oracle_softmax_causal_rows_f32(_fp(xs), M, N, ld, int(period), int(offset), _dp(y)) != 0:
        raise ValueError("oracle_softmax_causal_rows_f32 rejected its arguments")
    return y


def softmax_causal_rows_at(row, r: int, period: int, offset: int = 0) -> np.ndarray:
    """Causal softmax of one row standing at index r of the matrix: the row
    softmax of its kept prefix, 0 after it."""
    xr = _f64_row(row)
    kept = causal_kept(r, xr.size, period, offset)
    y = np.zeros_like(xr)
    if kept > 0:
        y[:kept] = softmax_row(xr[:kept])
    return y


def gelu_erf(z) -> np.ndarray:
    """Exact GELU 0.5 z (1 + erf(z / sqrt(2)))."""
    f = lib().oracle_gelu_erf
    zz = np.asarray(z, dtype=np.float64)
    return np.vectorize(f, otypes=[np.float64])(zz) if zz.ndim else np.float64(f(float(zz)))


def layernorm_gelu_erf(x, w=None, b=None, eps: float = 1e-5) -> np.ndarray:
    """LayerNorm -> affine -> exact GELU of every row -> float64 (M, N)."""
    xs, M, N, ld = _rows(x)
    y = np.empty((M, N), dtype=np.float64)
    wf, bf = _opt32(w, N), _opt32(b, N)
    if lib().oracle_layernorm_gelu_erf_rows_f32(_fp(xs), _fp(wf), _fp(bf), float(eps), M, N, ld, _dp(y)) != 0:
        raise ValueError("oracle_layernorm_gelu_erf_rows_f32 rejected its arguments")
    return y


def bias_residual_gelu(x, residual=None, bias=None, approximate: str = "none") -> np.ndarray:
    """GELU(x + bias + residual) of every element -> float64 (M, N); bias per
    column, residual shaped like x (either may be None); approximate "none"
    (exact, erf) or "tanh"."""
    if approximate not in ("none", "tanh"):
        raise ValueError('approximate must be "none" or "tanh"')
    xs, M, N, ld = _rows(x)
    rs = None
    if residual is not None:
        rs, Mr, Nr, ldr = _rows(residual)
        if (Mr, Nr) != (M, N):
            raise ValueError("residual must have x's shape")
        if ldr != ld:
            xs, rs, ld = np.ascontiguousarray(xs), np.ascontiguousarray(rs), N
    y = np.empty((M, N), dtype=np.float64)
    if lib().oracle_bias_residual_gelu_rows_f32(_fp(xs), _fp(rs), _fp(_opt32(bias, N)), M, N, ld,
                                                0 if approximate == "none" else 1, _dp(y)) != 0:
        raise ValueError("oracle_bias_residual_gelu_rows_f32 rejected its arguments")
    return y


def row_sum(x) -> np.ndarray:
    """Sum of every row -> float64 (M,)."""
    xs, M, N, ld = _rows(x)
    out = np.empty(M, dtype=np.float64)
    if lib().oracle_row_sum_rows_f32(_fp(xs), M, N, ld, _dp(out)) != 0:
        raise ValueError("oracle_row_sum_rows_f32 rejected its arguments")
    return out


def row_max(x) -> np.ndarray:
    """Maximum of every row -> float64 (M,) (NaN if the row holds a NaN)."""
    xs, M, N, ld = _rows(x)
    out = np.empty(M, dtype=np.float64)
    if lib().oracle_row_max_rows_f32(_fp(xs), M, N, ld, _dp(out)) != 0:
        raise ValueError("oracle_row_max_rows_f32 rejected its arguments")
    return out


def gelu_tanh_grad(z) -> np.ndarray:
    """d/dz of the tanh-approximation GELU."""
    f = lib().oracle_gelu_tanh_grad
    zz = np.asarray(z, dtype=np.float64)
    return np.vectorize(f, otypes=[np.float64])(zz) if zz.ndim else np.float64(f(float(zz)))


def layernorm_gelu_backward_row(x, dy, w=None, b=None, eps: float = 1e-5):
    """(dx, dw, db) of one row (dw, db for this row alone)."""
    xr, gr = _f64_row(x), _f64_row(dy)
    n = xr.size
    dx, dw, db = np.empty(n), np.zeros(n), np.zeros(n)
    lib().oracle_layernorm_gelu_backward_row(_dp(xr), _dp(gr), _dp(_opt64(w, n)), _dp(_opt64(b, n)), float(eps), n,
                                             _dp(dx), _dp(dw), _dp(db))
    return dx, dw, db


def layernorm_gelu_backward(x, dy, w=None, b=None, eps: float = 1e-5):
    """(dx (M, N), dw (N,), db (N,)) of the LayerNorm -> affine -> tanh-GELU backward."""
    xs, M, N, ld = _rows(x)
    gs, Mg, Ng, ldg = _rows(dy)
    if (Mg, Ng) != (M, N):
        raise ValueError("x and dy must have the same shape")
    if ldg != ld:
        xs, gs, ld = np.ascontiguousarray(xs), np.ascontiguousarray(gs), N
    dx = np.empty((M, N)); dw = np.empty(N); db = np.empty(N)
    if lib().oracle_layernorm_gelu_backward_rows_f32(_fp(xs), _fp(gs), _fp(_opt32(w, N)), _fp(_opt32(b, N)),
                                                     float(eps), M, N, ld, _dp(dx), _dp(dw), _dp(db)) != 0:
        raise ValueError("oracle_layernorm_gelu_backward_rows_f32 rejected its arguments")
    return dx, dw, db
