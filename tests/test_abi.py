"""C ABI checks that need no GPU: the library loads, exports every entry point
include/rowops.h declares, and rejects invalid arguments with the documented
status before any CUDA call (so these calls launch nothing)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rowops.h")

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3
F32, BF16 = 0, 1


@pytest.fixture(scope="module")
def lib():
    from row_wise_reduction_gb300 import build
    from row_wise_reduction_gb300.rowops import library

    build.build()
    return library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rowops_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("rowops_softmax", "rowops_online_softmax", "rowops_layernorm_gelu",
              "rowops_online_softmax_workspace_bytes", "rowops_online_softmax_status", "rowops_status_string",
              "rowops_rmsnorm", "rowops_fused_residual_rmsnorm", "rowops_softmax_causal", "rowops_row_sum",
              "rowops_row_max", "rowops_layernorm_gelu_erf", "rowops_gelu",
              "rowops_layernorm_gelu_backward", "rowops_layernorm_gelu_backward_workspace_bytes",
              "rowops_bias_residual_gelu"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(lib._name)
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} declared in rowops.h but not exported"


def test_status_strings(lib):
    for code, name in [(0, "ROWOPS_OK"), (1, "ROWOPS_ERR_INVALID_VALUE"), (2, "ROWOPS_ERR_UNSUPPORTED"),
                       (3, "ROWOPS_ERR_WORKSPACE"), (4, "ROWOPS_ERR_CUDA"), (5, "ROWOPS_ERR_TIMEOUT")]:
        assert lib.rowops_status_string(code).decode() == name
    assert lib.rowops_status_string(99).decode() == "ROWOPS_ERR_UNKNOWN"


X = 0x10000  # fake device addresses: validation fails before any use
Y = 0x90000


@pytest.mark.parametrize(
    "args,want",
    [
        ((X, Y, 4, 8, 8, 7, None), INVALID),  # bad dtype
        ((X, Y, -1, 8, 8, F32, None), INVALID),  # M < 0
        ((X, Y, 4, 0, 8, F32, None), INVALID),  # N < 1
        ((X, Y, 4, 8, 7, F32, None), INVALID),  # ld < N
        ((None, Y, 4, 8, 8, F32, None), INVALID),  # null x
        ((X, None, 4, 8, 8, F32, None), INVALID),  # null y
        ((X + 2, Y, 4, 8, 8, F32, None), INVALID),  # x not 4-byte aligned for fp32
        ((X, Y + 1, 4, 8, 8, BF16, None), INVALID),  # y not 2-byte aligned for bf16
        ((X, X + 16, 4, 8, 8, F32, None), INVALID),  # partial overlap
        ((X, Y, 4, 1 << 31, 1 << 31, F32, None), UNSUPPORTED),  # N too large
        ((X, Y, 1 << 62, 8, 1 << 40, F32, None), UNSUPPORTED),  # byte span overflows int64
        ((None, None, 0, 8, 8, F32, None), OK),  # M == 0: no-op, no CUDA call
    ],
)
def test_softmax_validation(lib, args, want):
    assert lib.rowops_softmax(*args) == want


def test_layernorm_gelu_validation(lib):
    f = lib.rowops_layernorm_gelu
    assert f(X, Y, None, None, -1.0, 4, 8, 8, F32, None) == INVALID  # eps < 0
    assert f(X, Y, None, None, float("nan"), 4, 8, 8, F32, None) == INVALID
    assert f(X, Y, None, None, float("inf"), 4, 8, 8, F32, None) == INVALID
    assert f(X, Y, X + 0x40001, None, 1e-5, 4, 8, 8, BF16, None) == INVALID  # misaligned w
    assert f(X, Y, None, Y + 0x40002, 1e-5, 4, 8, 8, F32, None) == INVALID  # misaligned b
    assert f(X, Y, None, None, 1e-5, 4, 8, 4, F32, None) == INVALID  # ld < N
    assert f(None, None, None, None, 1e-5, 0, 8, 8, F32, None) == OK


def test_softmax_causal_validation(lib):
    f = lib.rowops_softmax_causal
    assert f(X, Y, 4, 8, 8, 0, 0, F32, None) == INVALID  # period < 1
    assert f(X, Y, 4, 8, 8, -3, 0, F32, None) == INVALID
    assert f(X, Y, 4, 8, 8, 8, (1 << 62) + 1, F32, None) == INVALID  # offset out of range
    assert f(X, Y, 4, 8, 8, 8, -(1 << 62) - 1, F32, None) == INVALID
    assert f(X, X + 16, 4, 8, 8, 8, 0, F32, None) == INVALID  # partial overlap
    assert f(None, Y, 4, 8, 8, 8, 0, F32, None) == INVALID
    assert f(None, None, 0, 8, 8, 8, 0, F32, None) == OK


@pytest.mark.parametrize("fn", ["rowops_row_sum", "rowops_row_max"])
def test_row_reduction_validation(lib, fn):
    f = getattr(lib, fn)
    O = 0x700000
    assert f(X, None, 4, 8, 8, F32, None) == INVALID  # null out
    assert f(X, O + 2, 4, 8, 8, F32, None) == INVALID  # out not 4-byte aligned
    assert f(X, X + 8, 4, 8, 8, F32, None) == INVALID  # out overlaps the rows of x
    assert f(None, O, 4, 8, 8, F32, None) == INVALID
    assert f(X, O, 4, 8, 7, F32, None) == INVALID  # ld < N
    assert f(X + 1, O, 4, 8, 8, BF16, None) == INVALID  # x not 2-byte aligned
    assert f(None, None, 0, 8, 8, F32, None) == OK


def test_gelu_validation(lib):
    f = lib.rowops_gelu
    assert f(X, Y, 16, 2, F32, None) == INVALID  # approximate must be 0 or 1
    assert f(X, Y, -1, 0, F32, None) == INVALID
    assert f(X, X + 16, 16, 0, F32, None) == INVALID  # partial overlap
    assert f(None, Y, 16, 1, BF16, None) == INVALID
    assert f(X + 1, Y, 16, 1, BF16, None) == INVALID  # misaligned bf16
    assert f(None, None, 0, 0, F32, None) == OK
    g = lib.rowops_layernorm_gelu_erf
    assert g(X, Y, None, None, -1.0, 4, 8, 8, F32, None) == INVALID
    assert g(None, None, None, None, 1e-5, 0, 8, 8, F32, None) == OK


def test_rmsnorm_validation(lib):
    f = lib.rowops_rmsnorm
    assert f(X, Y, None, -1.0, 4, 8, 8, F32, None) == INVALID  # eps < 0
    assert f(X, Y, None, float("nan"), 4, 8, 8, F32, None) == INVALID
    assert f(X, Y, X + 0x40001, 1e-5, 4, 8, 8, BF16, None) == INVALID  # misaligned w
    assert f(X, X + 16, None, 1e-5, 4, 8, 8, F32, None) == INVALID  # partial overlap
    assert f(None, Y, None, 1e-5, 4, 8, 8, F32, None) == INVALID
    assert f(X, Y, None, 1e-5, 4, 8, 8, 5, None) == INVALID  # bad dtype
    assert f(None, None, None, 1e-5, 0, 8, 8, F32, None) == OK


R, RO = 0x200000, 0x300000


def test_fused_residual_rmsnorm_validation(lib):
    f = lib.rowops_fused_residual_rmsnorm
    args = lambda x=X, r=R, y=Y, ro=RO, w=None, eps=1e-5, M=4, N=8, ld=8, dt=F32: (x, r, y, ro, w, eps, M, N, ld, dt,
                                                                                  None)
    assert f(*args(r=None)) == INVALID  # null residual
    assert f(*args(ro=None)) == INVALID  # null residual_out
    assert f(*args(eps=-1.0)) == INVALID
    assert f(*args(y=RO)) == INVALID  # y and residual_out are the same memory
    assert f(*args(y=RO + 64)) == INVALID  # y overlaps residual_out
    assert f(*args(ro=X + 16)) == INVALID  # residual_out partly overlaps x
    assert f(*args(y=R + 32)) == INVALID  # y partly overlaps residual
    assert f(*args(w=X + 0x40002, dt=F32)) == INVALID  # misaligned w
    assert f(*args(ro=R + 1, dt=BF16)) == INVALID  # misaligned residual_out
    assert f(*args(N=1 << 31, ld=1 << 31)) == UNSUPPORTED
    assert f(None, None, None, None, None, 1e-5, 0, 8, 8, F32, None) == OK


def test_online_softmax_workspace_bytes(lib):
    q = lib.rowops_online_softmax_workspace_bytes
    # header, M 64-bit row results padded to 256 bytes, M * (ceil(N / 256) + 2) 8-byte partials
    assert q(64, 1 << 20, F32) == 256 + 512 + 64 * 4098 * 8
    assert q(3, 1, BF16) == 256 + 256 + 3 * 3 * 8
    assert q(5, 257, F32) == 256 + 256 + 5 * 4 * 8
    assert q(33, 257, F32) == 256 + 512 + 33 * 4 * 8
    assert q(0, 100, F32) == 256
    assert q(-1, 100, F32) == 0
    assert q(4, 0, F32) == 0
    assert q(4, 100, 9) == 0


def test_online_softmax_validation(lib):
    f = lib.rowops_online_softmax
    need = lib.rowops_online_softmax_workspace_bytes(4, 1000, F32)
    WS = 0x200000
    assert f(X, Y, 4, 1000, 1000, F32, None, need, 0, None) == WORKSPACE
    assert f(X, Y, 4, 1000, 1000, F32, WS + 16, need, 0, None) == WORKSPACE  # not 256-byte aligned
    assert f(X, Y, 4, 1000, 1000, F32, WS, need - 1, 0, None) == WORKSPACE
    for bad_chunk in (-16, 16, 255, 1000, 1 << 31):
        assert f(X, Y, 4, 1000, 1000, F32, WS, need, bad_chunk, None) == INVALID
    assert f(X, Y, 4, 1000, 999, F32, WS, need, 0, None) == INVALID
    assert f(None, None, 0, 1000, 1000, F32, None, 0, 0, None) == OK
    assert lib.rowops_online_softmax_status(None, None) == WORKSPACE


def test_layernorm_gelu_backward_workspace_bytes(lib):
    q = lib.rowops_layernorm_gelu_backward_workspace_bytes
    # dw, db partials (N floats each) of at most clamp(2^22 / N, 152, 4096) CTAs
    assert q(4, 8, F32) == 4096 * 2 * 8 * 4
    assert q(1 << 20, 8192, BF16) == 512 * 2 * 8192 * 4
    assert q(9, 768, F32) == 4096 * 2 * 768 * 4
    assert q(9, 4097, F32) == 1023 * 2 * 4097 * 4
    assert q(9, 1 << 20, F32) == 152 * 2 * (1 << 20) * 4
    assert q(0, 3, F32) == 4096 * 2 * 3 * 4
    assert q(-1, 8, F32) == 0
    assert q(4, 0, F32) == 0
    assert q(4, 8, 9) == 0


def test_layernorm_gelu_backward_validation(lib):
    f = lib.rowops_layernorm_gelu_backward
    DY, DW, DB, WS = 0x300000, 0x500000, 0x510000, 0x1000000
    need = lib.rowops_layernorm_gelu_backward_workspace_bytes(4, 8, F32)

    def args(x=X, dy=DY, w=None, b=None, eps=1e-5, dx=Y, dw=DW, db=DB, M=4, N=8, ld=8, dt=F32, ws=WS, nb=None):
        return (x, dy, w, b, eps, dx, dw, db, M, N, ld, dt, ws, need if nb is None else nb, None)

    assert f(*args(eps=-1.0)) == INVALID
    assert f(*args(eps=float("inf"))) == INVALID
    assert f(*args(eps=float("nan"))) == INVALID
    assert f(*args(dw=None)) == INVALID
    assert f(*args(db=DB + 2)) == INVALID  # db not 4-byte aligned
    assert f(*args(db=DW)) == INVALID  # dw and db the same
    assert f(*args(db=DW + 16)) == INVALID  # dw and db overlap
    assert f(*args(ws=None)) == WORKSPACE
    assert f(*args(ws=WS + 64)) == WORKSPACE  # not 256-byte aligned
    assert f(*args(nb=need - 1)) == WORKSPACE
    assert f(*args(dw=WS + 1024)) == INVALID  # dw inside the workspace
    assert f(*args(dx=X)) == INVALID  # dx must not alias x
    assert f(*args(dx=DY)) == INVALID  # nor dy
    assert f(*args(dx=DY + 16)) == INVALID
    assert f(*args(dy=None)) == INVALID
    assert f(*args(w=X + 0x40001, dt=BF16)) == INVALID  # misaligned w
    assert f(*args(b=X + 0x40001, dt=BF16)) == INVALID  # misaligned b
    assert f(*args(ld=7)) == INVALID
    assert f(*args(dt=5)) == INVALID


def test_bias_residual_gelu_validation(lib):
    f = lib.rowops_bias_residual_gelu
    R, BI = 0x300000, 0x500000

    def args(x=X, r=R, b=BI, y=Y, M=4, N=8, ld=8, ap=0, dt=F32):
        return (x, r, b, y, M, N, ld, ap, dt, None)

    assert f(*args(ap=2)) == INVALID
    assert f(*args(ap=-1)) == INVALID
    assert f(*args(x=None)) == INVALID
    assert f(*args(y=X + 16)) == INVALID  # y partly overlaps x
    assert f(*args(y=R + 16)) == INVALID  # y partly overlaps the residual
    assert f(*args(b=Y + 8)) == INVALID  # bias inside y's rows
    assert f(*args(b=BI + 2)) == INVALID  # bias not 4-byte aligned for fp32
    assert f(*args(r=R + 1, dt=BF16)) == INVALID  # residual not 2-byte aligned
    assert f(*args(ld=7)) == INVALID
    assert f(*args(dt=3)) == INVALID
    assert f(*args(N=1 << 31, ld=1 << 31)) == UNSUPPORTED
    assert f(*args(M=0)) == OK  # no rows: nothing to do, no CUDA call


def test_binding_has_no_fallback(monkeypatch, tmp_path):
    """The Python binding raises when the library is absent instead of
    computing anything itself."""
    import row_wise_reduction_gb300.rowops as r

    monkeypatch.setattr(r, "_lib", None)
    monkeypatch.setattr(r, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        r.library()


def test_call_module_marshals_like_ctypes(lib):
    """The binding's CPython call module passes the same arguments to the same
    entry points as ctypes: identical statuses on the validation cases (none
    of which reaches the GPU)."""
    from row_wise_reduction_gb300 import rowops as r

    r.library()
    fast = r._calls.module
    if fast is None:
        pytest.skip("the call module was not built (no gcc or Python headers)")
    for args in [(X, Y, 4, 8, 8, 7, None), (X, Y, 4, 0, 8, F32, None), (None, Y, 4, 8, 8, F32, None),
                 (X, X + 16, 4, 8, 8, F32, None), (X, Y, 1 << 62, 8, 1 << 40, F32, None),
                 (None, None, 0, 8, 8, F32, None)]:
        assert fast.softmax(*args) == lib.rowops_softmax(*args)
    for f, g in [(fast.layernorm_gelu, lib.rowops_layernorm_gelu), (fast.layernorm_gelu_erf,
                                                                     lib.rowops_layernorm_gelu_erf)]:
        for args in [(X, Y, None, None, -1.0, 4, 8, 8, F32, None), (X, Y, None, None, float("nan"), 4, 8, 8, F32, None),
                     (X, Y, X + 0x40001, None, 1e-5, 4, 8, 8, BF16, None), (X, Y, None, None, 1e-5, 4, 8, 4, F32, None),
                     (None, None, None, None, 1e-5, 0, 8, 8, F32, None)]:
            assert f(*args) == g(*args)
    with pytest.raises(TypeError):
        fast.softmax(X, Y, 4, 8, 8)


def test_binding_calls_through_ctypes_without_the_call_module(lib, monkeypatch):
    """Where the CPython call module is absent, the three launch-bound entry
    points bind to the library's ctypes functions instead: the same native
    code, never a Python computation."""
    import builtins

    from row_wise_reduction_gb300 import rowops as r

    real_import = builtins.__import__

    def no_call_module(name, *args, **kwargs):
        if name.endswith("_rowops_call") or (args and args[2] and "_rowops_call" in args[2]):
            raise ImportError("no call module")
        return real_import(name, *args, **kwargs)

    saved = r._calls
    monkeypatch.setattr(builtins, "__import__", no_call_module)
    try:
        r._bind_calls(r.library())
        c = r._calls
        assert c.module is None
        assert c.softmax is lib.rowops_softmax or c.softmax.__name__ == "rowops_softmax"
        assert c.softmax(None, None, 0, 8, 8, F32, None) == OK
        assert c.layernorm_gelu(X, Y, None, None, -1.0, 4, 8, 8, F32, None) == INVALID
    finally:
        monkeypatch.setattr(builtins, "__import__", real_import)
        r._calls = saved
