"""Python binding of librowops.so (argument marshalling only).

Each function has the name of the C entry point it calls and does no
arithmetic of its own: it checks shapes, takes device pointers, the row stride
and the current CUDA stream from torch tensors, calls the C ABI through
ctypes and raises :class:`RowopsError` on a non-OK status. PyTorch only
supplies device memory and streams. There is no CPU fallback: if the library
is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build import LIB as _LIB_PATH

__all__ = [
    "RowopsError",
    "library",
    "library_path",
    "rowops_softmax",
    "rowops_softmax_causal",
    "rowops_row_sum",
    "rowops_row_max",
    "rowops_online_softmax",
    "rowops_online_softmax_workspace_bytes",
    "rowops_online_softmax_status",
    "rowops_online_softmax_noalloc",
    "rowops_device_status",
    "rowops_layernorm_gelu",
    "rowops_layernorm_gelu_erf",
    "rowops_layernorm_gelu_backward",
    "rowops_layernorm_gelu_backward_workspace_bytes",
    "rowops_gelu",
    "rowops_bias_residual_gelu",
    "rowops_rmsnorm",
    "rowops_fused_residual_rmsnorm",
    "rowops_status_string",
    "rowops_reload_tuning",
    "ROWOPS_F32",
    "ROWOPS_BF16",
    "STATUS",
]

ROWOPS_F32 = 0
ROWOPS_BF16 = 1
STATUS = {
    0: "ROWOPS_OK",
    1: "ROWOPS_ERR_INVALID_VALUE",
    2: "ROWOPS_ERR_UNSUPPORTED",
    3: "ROWOPS_ERR_WORKSPACE",
    4: "ROWOPS_ERR_CUDA",
    5: "ROWOPS_ERR_TIMEOUT",
}

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64


class RowopsError(RuntimeError):
    """A rowops entry point returned a status other than ROWOPS_OK."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")


_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _LIB_PATH


def library() -> ctypes.CDLL:
    """Load librowops.so (built in-tree by ``row_wise_reduction_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with `python -m row_wise_reduction_gb300.build` "
                "(there is no fallback implementation)"
            )
        L = ctypes.CDLL(_LIB_PATH)
        L.rowops_status_string.restype = ctypes.c_char_p
        L.rowops_status_string.argtypes = [ctypes.c_int]
        L.rowops_reload_tuning.restype = None
        L.rowops_reload_tuning.argtypes = []
        L.rowops_softmax.restype = ctypes.c_int
        L.rowops_softmax.argtypes = [_vp, _vp, _i64, _i64, _i64, ctypes.c_int, _vp]
        L.rowops_online_softmax_workspace_bytes.restype = ctypes.c_size_t
        L.rowops_online_softmax_workspace_bytes.argtypes = [_i64, _i64, ctypes.c_int]
        L.rowops_online_softmax.restype = ctypes.c_int
        L.rowops_online_softmax.argtypes = [_vp, _vp, _i64, _i64, _i64, ctypes.c_int, _vp, ctypes.c_size_t,
                                            _i64, _vp]
        L.rowops_online_softmax_status.restype = ctypes.c_int
        L.rowops_online_softmax_status.argtypes = [_vp, _vp]
        L.rowops_device_status.restype = ctypes.c_int
        L.rowops_device_status.argtypes = [_vp]
        L.rowops_online_softmax_noalloc.restype = ctypes.c_int
        L.rowops_online_softmax_noalloc.argtypes = [_vp, _vp, _i64, _i64, _i64, ctypes.c_int, _i64, _vp]
        L.rowops_layernorm_gelu.restype = ctypes.c_int
        L.rowops_layernorm_gelu.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_float, _i64, _i64, _i64,
                                            ctypes.c_int, _vp]
        for name in ("rowops_row_sum", "rowops_row_max"):
            getattr(L, name).restype = ctypes.c_int
            getattr(L, name).argtypes = [_vp, _vp, _i64, _i64, _i64, ctypes.c_int, _vp]
        L.rowops_softmax_causal.restype = ctypes.c_int
        L.rowops_softmax_causal.argtypes = [_vp, _vp, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, _vp]
        L.rowops_layernorm_gelu_erf.restype = ctypes.c_int
        L.rowops_layernorm_gelu_erf.argtypes = L.rowops_layernorm_gelu.argtypes
        L.rowops_gelu.restype = ctypes.c_int
        L.rowops_gelu.argtypes = [_vp, _vp, _i64, ctypes.c_int, ctypes.c_int, _vp]
        L.rowops_rmsnorm.restype = ctypes.c_int
        L.rowops_rmsnorm.argtypes = [_vp, _vp, _vp, ctypes.c_float, _i64, _i64, _i64, ctypes.c_int, _vp]
        L.rowops_fused_residual_rmsnorm.restype = ctypes.c_int
        L.rowops_fused_residual_rmsnorm.argtypes = [_vp, _vp, _vp, _vp, _vp, ctypes.c_float, _i64, _i64, _i64,
                                                    ctypes.c_int, _vp]
        L.rowops_bias_residual_gelu.restype = ctypes.c_int
        L.rowops_bias_residual_gelu.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int,
                                                _vp]
        L.rowops_layernorm_gelu_backward_workspace_bytes.restype = ctypes.c_size_t
        L.rowops_layernorm_gelu_backward_workspace_bytes.argtypes = [_i64, _i64, ctypes.c_int]
        L.rowops_layernorm_gelu_backward.restype = ctypes.c_int
        L.rowops_layernorm_gelu_backward.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _i64,
                                                     _i64, _i64, ctypes.c_int, _vp, ctypes.c_size_t, _vp]
        _bind_calls(L)  # before _lib: a thread that sees _lib set finds _calls set too
        _lib = L
    return _lib


class _Calls:
    """The entry points whose small calls are bound by host time: through the
    CPython call module ``_rowops_call`` where it was built (about 0.1 us of
    marshalling per call), else through ctypes (about 2 us)."""

    __slots__ = ("softmax", "layernorm_gelu", "layernorm_gelu_erf", "module")


_calls: Optional[_Calls] = None


def _bind_calls(L: ctypes.CDLL) -> None:
    global _calls
    c = _Calls()
    try:
        from . import _rowops_call as fast
    except ImportError:
        fast = None
    if fast is not None:
        def addr(f):
            return ctypes.cast(f, ctypes.c_void_p).value

        fast.bind(addr(L.rowops_softmax), addr(L.rowops_layernorm_gelu), addr(L.rowops_layernorm_gelu_erf))
        c.softmax, c.layernorm_gelu, c.layernorm_gelu_erf = fast.softmax, fast.layernorm_gelu, fast.layernorm_gelu_erf
    else:
        c.softmax, c.layernorm_gelu, c.layernorm_gelu_erf = (L.rowops_softmax, L.rowops_layernorm_gelu,
                                                              L.rowops_layernorm_gelu_erf)
    c.module = fast
    _calls = c


def _hot_calls() -> _Calls:
    library()
    return _calls


def rowops_status_string(status: int) -> str:
    return library().rowops_status_string(int(status)).decode()


def rowops_reload_tuning() -> None:
    """Make the library read the ROWOPS_* knobs from the environment again
    (it reads them once, at its first call, otherwise)."""
    library().rowops_reload_tuning()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return ROWOPS_F32
    if t.dtype == torch.bfloat16:
        return ROWOPS_BF16
    raise TypeError(f"rowops supports float32 and bfloat16, not {t.dtype}")


def _rows(t: torch.Tensor, name: str):
    """(M, N, ld) of a 2-D CUDA tensor with unit column stride. (Each tensor
    property is read once: at the small, launch-bound sizes the binding's own
    checks are a visible share of a call.)"""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    sh = t.shape
    if len(sh) != 2:
        raise ValueError(f"{name} must be 2-D (M, N)")
    M, N = sh
    st = t.stride()
    if N > 0 and st[1] != 1:
        raise ValueError(f"{name} must have unit column stride")
    return M, N, (st[0] if M > 1 else max(N, st[0]))


def _out_like(x: torch.Tensor, y: Optional[torch.Tensor]) -> torch.Tensor:
    if y is None:
        return torch.empty_strided(x.shape, x.stride(), dtype=x.dtype, device=x.device)
    if y.dtype is not x.dtype or y.get_device() != x.get_device() or y.shape != x.shape:
        raise ValueError("y must match x in shape, dtype and device")
    if y.shape[0] > 1 and y.stride() != x.stride():
        raise ValueError("x and y must share the row stride")
    return y


_current_device = getattr(torch._C, "_cuda_getDevice", None) or torch.cuda.current_device
_current_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device=None) -> int:
    if stream is None:
        # the raw handle of the current device's current stream (the cheap
        # form of torch.cuda.current_stream().cuda_stream; the tensors passed
        # in are CUDA tensors, so CUDA is initialised already)
        return _current_raw_stream(_current_device() if device is None else device)
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


_DTYPE_CODES = {torch.float32: ROWOPS_F32, torch.bfloat16: ROWOPS_BF16}


def _xy(x: torch.Tensor, y: Optional[torch.Tensor]):
    """_rows(x) and _out_like(x, y) in one pass over the tensors' properties,
    for the entry points whose small calls are bound by host time: returns
    (M, N, ld, y, dtype code, device index)."""
    sh = x.shape
    if len(sh) != 2:
        raise ValueError("x must be 2-D (M, N)")
    dev = x.get_device()
    if dev < 0:
        raise ValueError("x must be a CUDA tensor")
    M, N = sh
    st = x.stride()
    if N > 0 and st[1] != 1:
        raise ValueError("x must have unit column stride")
    dt = x.dtype
    code = _DTYPE_CODES.get(dt)
    if code is None:
        raise TypeError(f"rowops supports float32 and bfloat16, not {dt}")
    if y is None:
        y = torch.empty_strided(sh, st, dtype=dt, device=x.device)
    else:
        if y.dtype is not dt or y.get_device() != dev or y.shape != sh:
            raise ValueError("y must match x in shape, dtype and device")
        if M > 1 and y.stride() != st:
            raise ValueError("x and y must share the row stride")
    return M, N, (st[0] if M > 1 else max(N, st[0])), y, code, dev


def _check(fn: str, status: int):
    if status != 0:
        raise RowopsError(fn, status)


def rowops_softmax(x: torch.Tensor, y: Optional[torch.Tensor] = None, *, stream=None) -> torch.Tensor:
    """Stable softmax of every row of ``x`` (M, N) into ``y`` (may be ``x``)."""
    M, N, ld, y, code, dev = _xy(x, y)
    st = (_calls or _hot_calls()).softmax(x.data_ptr(), y.data_ptr(), M, N, ld, code,
                                          _current_raw_stream(dev) if stream is None else _stream(stream))
    if st:
        raise RowopsError("rowops_softmax", st)
    return y


def rowops_online_softmax_workspace_bytes(M: int, N: int, dtype: torch.dtype) -> int:
    code = ROWOPS_F32 if dtype == torch.float32 else ROWOPS_BF16 if dtype == torch.bfloat16 else -1
    return int(library().rowops_online_softmax_workspace_bytes(int(M), int(N), code))


def rowops_online_softmax(
    x: torch.Tensor,
    y: Optional[torch.Tensor] = None,
    *,
    workspace: Optional[torch.Tensor] = None,
    chunk: int = 0,
    stream=None,
) -> torch.Tensor:
    """Split-row online softmax of every row of ``x``.

    ``workspace``: a CUDA uint8 tensor of at least
    ``rowops_online_softmax_workspace_bytes(M, N, dtype)`` bytes; allocated
    here when omitted. ``chunk``: columns per CTA chunk (0 = automatic).
    """
    M, N, ld = _rows(x, "x")
    y = _out_like(x, y)
    need = rowops_online_softmax_workspace_bytes(M, N, x.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    if not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    st = library().rowops_online_softmax(x.data_ptr(), y.data_ptr(), M, N, ld, _dtype_code(x),
                                         workspace.data_ptr(), nbytes, int(chunk), _stream(stream))
    _check("rowops_online_softmax", st)
    return y


def rowops_online_softmax_status(workspace: torch.Tensor, *, stream=None) -> int:
    """Synchronise the stream and return the device-side status of the last
    rowops_online_softmax call on ``workspace`` (0 = ROWOPS_OK)."""
    return int(library().rowops_online_softmax_status(workspace.data_ptr(), _stream(stream)))


def rowops_device_status(*, stream=None) -> int:
    """Synchronise the stream, then read and clear the library's device error
    word on the current device (0 = ROWOPS_OK, 5 = a bounded device-side wait
    gave up)."""
    return int(library().rowops_device_status(_stream(stream)))


def rowops_online_softmax_noalloc(
    x: torch.Tensor, y: Optional[torch.Tensor] = None, *, chunk: int = 0, stream=None
) -> torch.Tensor:
    """rowops_online_softmax without a workspace, for callers that cannot
    allocate device memory: the partials live in the library's own 1 MiB
    device array (M * ceil(N / chunk) <= 131040). Calls that could overlap on
    the GPU share that array and must be ordered."""
    M, N, ld = _rows(x, "x")
    y = _out_like(x, y)
    st = library().rowops_online_softmax_noalloc(x.data_ptr(), y.data_ptr(), M, N, ld, _dtype_code(x), int(chunk),
                                                 _stream(stream))
    _check("rowops_online_softmax_noalloc", st)
    return y


def rowops_layernorm_gelu(
    x: torch.Tensor,
    w: Optional[torch.Tensor] = None,
    b: Optional[torch.Tensor] = None,
    eps: float = 1e-5,
    y: Optional[torch.Tensor] = None,
    *,
    stream=None,
) -> torch.Tensor:
    """Fused LayerNorm -> affine -> tanh-GELU of every row of ``x``."""
    M, N, ld, y, code, dev = _xy(x, y)
    st = (_calls or _hot_calls()).layernorm_gelu(
        x.data_ptr(), y.data_ptr(), _affine(w, x, N, dev, "w"), _affine(b, x, N, dev, "b"), float(eps), M, N, ld,
        code, _current_raw_stream(dev) if stream is None else _stream(stream))
    if st:
        raise RowopsError("rowops_layernorm_gelu", st)
    return y


def rowops_layernorm_gelu_erf(
    x: torch.Tensor,
    w: Optional[torch.Tensor] = None,
    b: Optional[torch.Tensor] = None,
    eps: float = 1e-5,
    y: Optional[torch.Tensor] = None,
    *,
    stream=None,
) -> torch.Tensor:
    """Fused LayerNorm -> affine -> exact (erf) GELU of every row of ``x``."""
    M, N, ld, y, code, dev = _xy(x, y)
    st = (_calls or _hot_calls()).layernorm_gelu_erf(
        x.data_ptr(), y.data_ptr(), _affine(w, x, N, dev, "w"), _affine(b, x, N, dev, "b"), float(eps), M, N, ld,
        code, _current_raw_stream(dev) if stream is None else _stream(stream))
    if st:
        raise RowopsError("rowops_layernorm_gelu_erf", st)
    return y


def rowops_layernorm_gelu_backward_workspace_bytes(M: int, N: int, dtype: torch.dtype) -> int:
    code = ROWOPS_F32 if dtype == torch.float32 else ROWOPS_BF16 if dtype == torch.bfloat16 else -1
    return int(library().rowops_layernorm_gelu_backward_workspace_bytes(int(M), int(N), code))


def _grad_out(t: Optional[torch.Tensor], N: int, device, name: str) -> torch.Tensor:
    if t is None:
        return torch.empty(N, dtype=torch.float32, device=device)
    if t.dtype != torch.float32 or t.numel() != N or not t.is_contiguous() or t.device != device:
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of N entries")
    return t


def rowops_layernorm_gelu_backward(
    x: torch.Tensor,
    dy: torch.Tensor,
    w: Optional[torch.Tensor] = None,
    b: Optional[torch.Tensor] = None,
    eps: float = 1e-5,
    dx: Optional[torch.Tensor] = None,
    dw: Optional[torch.Tensor] = None,
    db: Optional[torch.Tensor] = None,
    workspace: Optional[torch.Tensor] = None,
    *,
    stream=None,
):
    """Gradients of rowops_layernorm_gelu (tanh GELU) for the upstream gradient
    ``dy``: returns ``(dx, dw, db)``, dx in x's dtype and layout, dw and db
    float32 (N,). ``workspace``: a CUDA uint8 tensor of at least
    ``rowops_layernorm_gelu_backward_workspace_bytes(M, N, dtype)`` bytes,
    allocated per call when omitted."""
    M, N, ld = _rows(x, "x")
    _out_like(x, dy)  # same shape, dtype, device and row stride
    dx = _out_like(x, dx)
    pw, pb = _weight(w, x, N, "w"), _weight(b, x, N, "b")
    dw = _grad_out(dw, N, x.device, "dw")
    db = _grad_out(db, N, x.device, "db")
    need = rowops_layernorm_gelu_backward_workspace_bytes(M, N, x.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    if not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    nbytes = workspace.numel() * workspace.element_size()
    st = library().rowops_layernorm_gelu_backward(
        x.data_ptr(), dy.data_ptr(), pw, pb, float(eps), dx.data_ptr(), dw.data_ptr(), db.data_ptr(), M, N, ld,
        _dtype_code(x), workspace.data_ptr(), nbytes, _stream(stream))
    _check("rowops_layernorm_gelu_backward", st)
    return dx, dw, db


def rowops_bias_residual_gelu(
    x: torch.Tensor,
    residual: Optional[torch.Tensor] = None,
    bias: Optional[torch.Tensor] = None,
    y: Optional[torch.Tensor] = None,
    approximate: str = "none",
    *,
    stream=None,
) -> torch.Tensor:
    """y = GELU(x + bias + residual) for every row of ``x`` (bias per column;
    residual shaped and strided like x; either may be None); approximate
    "none" (exact, erf) or "tanh"."""
    if approximate not in ("none", "tanh"):
        raise ValueError('approximate must be "none" or "tanh"')
    M, N, ld = _rows(x, "x")
    if residual is not None:
        _out_like(x, residual)  # same shape, dtype, device and row stride
    y = _out_like(x, y)
    st = library().rowops_bias_residual_gelu(
        x.data_ptr(), residual.data_ptr() if residual is not None else None, _weight(bias, x, N, "bias"),
        y.data_ptr(), M, N, ld, 0 if approximate == "none" else 1, _dtype_code(x), _stream(stream))
    _check("rowops_bias_residual_gelu", st)
    return y


def _affine(v: Optional[torch.Tensor], x: torch.Tensor, N: int, dev: int, name: str):
    """Device pointer of an optional per-column vector (w, b) of x's dtype."""
    if v is None:
        return None
    if v.dtype is not x.dtype or v.get_device() != dev or v.numel() != N or not v.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor of N entries with x's dtype")
    return v.data_ptr()


def _weight(w: Optional[torch.Tensor], x: torch.Tensor, N: int, name: str = "w"):
    if w is None:
        return None
    if w.dtype != x.dtype or w.device != x.device or w.numel() != N or not w.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor of N entries with x's dtype")
    return w.data_ptr()


def rowops_rmsnorm(
    x: torch.Tensor,
    w: Optional[torch.Tensor] = None,
    eps: float = 1e-5,
    y: Optional[torch.Tensor] = None,
    *,
    stream=None,
) -> torch.Tensor:
    """RMSNorm of every row of ``x``: x * rsqrt(mean(x^2) + eps) * w."""
    M, N, ld = _rows(x, "x")
    y = _out_like(x, y)
    st = library().rowops_rmsnorm(x.data_ptr(), y.data_ptr(), _weight(w, x, N), float(eps), M, N, ld,
                                  _dtype_code(x), _stream(stream))
    _check("rowops_rmsnorm", st)
    return y


def rowops_fused_residual_rmsnorm(
    x: torch.Tensor,
    residual: torch.Tensor,
    w: Optional[torch.Tensor] = None,
    eps: float = 1e-5,
    y: Optional[torch.Tensor] = None,
    residual_out: Optional[torch.Tensor] = None,
    *,
    stream=None,
):
    """residual_out = x + residual and y = RMSNorm(residual_out) * w, in one
    pass; returns ``(y, residual_out)``. Outputs may be given (e.g.
    ``residual_out=residual`` to update the residual stream in place)."""
    M, N, ld = _rows(x, "x")
    _out_like(x, residual)  # same shape, dtype, device and row stride
    y = _out_like(x, y)
    residual_out = _out_like(x, residual_out)
    st = library().rowops_fused_residual_rmsnorm(
        x.data_ptr(), residual.data_ptr(), y.data_ptr(), residual_out.data_ptr(), _weight(w, x, N), float(eps),
        M, N, ld, _dtype_code(x), _stream(stream))
    _check("rowops_fused_residual_rmsnorm", st)
    return y, residual_out


def rowops_softmax_causal(
    x: torch.Tensor,
    period: Optional[int] = None,
    offset: int = 0,
    y: Optional[torch.Tensor] = None,
    *,
    stream=None,
) -> torch.Tensor:
    """Causal softmax: row r keeps the columns c <= (r mod period) + offset
    (default period: N, the stacked square causal masks); masked columns are
    not read and come out 0."""
    M, N, ld = _rows(x, "x")
    y = _out_like(x, y)
    period = N if period is None else int(period)
    st = library().rowops_softmax_causal(x.data_ptr(), y.data_ptr(), M, N, ld, period, int(offset),
                                         _dtype_code(x), _stream(stream))
    _check("rowops_softmax_causal", st)
    return y


def _row_reduce(fn: str, x: torch.Tensor, out: Optional[torch.Tensor], stream) -> torch.Tensor:
    M, N, ld = _rows(x, "x")
    if out is None:
        out = torch.empty(M, dtype=torch.float32, device=x.device)
    elif out.dtype != torch.float32 or out.numel() != M or not out.is_contiguous() or out.device != x.device:
        raise ValueError("out must be a contiguous float32 CUDA tensor of M entries")
    st = getattr(library(), fn)(x.data_ptr(), out.data_ptr(), M, N, ld, _dtype_code(x), _stream(stream))
    _check(fn, st)
    return out


def rowops_row_sum(x: torch.Tensor, out: Optional[torch.Tensor] = None, *, stream=None) -> torch.Tensor:
    """Sum of every row of ``x`` as float32 (M,)."""
    return _row_reduce("rowops_row_sum", x, out, stream)


def rowops_row_max(x: torch.Tensor, out: Optional[torch.Tensor] = None, *, stream=None) -> torch.Tensor:
    """Maximum of every row of ``x`` as float32 (M,); NaN where a row holds a NaN."""
    return _row_reduce("rowops_row_max", x, out, stream)


def rowops_gelu(x: torch.Tensor, y: Optional[torch.Tensor] = None, approximate: str = "none", *,
                stream=None) -> torch.Tensor:
    """Elementwise GELU of a contiguous tensor: approximate "none" (exact, erf)
    or "tanh"."""
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor")
    if approximate not in ("none", "tanh"):
        raise ValueError('approximate must be "none" or "tanh"')
    if y is None:
        y = torch.empty_like(x)
    elif y.shape != x.shape or y.dtype != x.dtype or y.device != x.device or not y.is_contiguous():
        raise ValueError("y must be a contiguous tensor matching x")
    st = library().rowops_gelu(x.data_ptr(), y.data_ptr(), x.numel(), 0 if approximate == "none" else 1,
                               _dtype_code(x), _stream(stream))
    _check("rowops_gelu", st)
    return y
