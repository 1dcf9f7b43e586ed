"""Pins for the CPU oracle: closed forms, invariants, exact-arithmetic brute
force and library routines, so that the oracle is checked against something
other than itself before it is used to check the CUDA path.

Each test names the mistake it would catch. Nothing here needs a GPU.
"""
import decimal
import math
from decimal import Decimal

import numpy as np
import pytest
import torch

from tests import _golden

CTX = decimal.Context(prec=60)


# ----------------------------------------------------------------------------
# exact-arithmetic brute force (Decimal, 60 digits), independent of the oracle
# ----------------------------------------------------------------------------
def _dec(v: float) -> Decimal:
    return Decimal(v)  # exact conversion of the double


def bf_softmax(xs):
    xd = [_dec(v) for v in xs]
    m = max(xd)
    e = [CTX.exp(CTX.subtract(v, m)) for v in xd]
    s = sum(e, Decimal(0))
    return [float(CTX.divide(v, s)) for v in e]


def bf_tanh(u: Decimal) -> Decimal:
    if u < 0:
        return -bf_tanh(-u)
    t = CTX.exp(CTX.multiply(Decimal(-2), u))
    return CTX.divide(1 - t, 1 + t)


def bf_gelu(z: float, k0=Decimal("0.79788456"), k1=Decimal("0.044715")) -> float:
    zd = _dec(z)
    inner = CTX.multiply(k0, zd + CTX.multiply(k1, CTX.power(zd, 3)))
    return float(CTX.multiply(CTX.multiply(Decimal("0.5"), zd), 1 + bf_tanh(inner)))


def bf_layernorm(xs, w=None, b=None, eps=1e-5):
    xd = [_dec(v) for v in xs]
    n = len(xd)
    mean = CTX.divide(sum(xd, Decimal(0)), n)
    var = CTX.divide(sum((CTX.subtract(v, mean) ** 2 for v in xd), Decimal(0)), n)
    rstd = CTX.divide(1, CTX.sqrt(var + _dec(eps)))
    out = []
    for j, v in enumerate(xd):
        wj = _dec(w[j]) if w is not None else Decimal(1)
        bj = _dec(b[j]) if b is not None else Decimal(0)
        out.append(CTX.multiply(CTX.multiply(v - mean, rstd), wj) + bj)
    return out


def _rng(seed):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------------------
# softmax
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("case", _golden.read_cases("softmax_closed_forms.txt"), ids=lambda c: c[0])
def test_softmax_golden_closed_forms(oracle, case):
    """Worked examples: catches a wrong normaliser, a missing max subtraction
    (large_shift case overflows exp without it), -inf handling and the
    all-masked convention."""
    _, _, rows = case
    x = [float(v) for v in rows["x"]]
    want = [float(v) for v in rows["y"]]
    # rounding x_j to double moves exp(x_j - m) by up to |x_j| 2^-52 relative
    finite = [abs(v) for v in x if math.isfinite(v)]
    rtol = 2e-15 + 2.0 ** -51 * max(finite, default=0.0)
    outs = [oracle.softmax_row(x)]
    # the online and split forms reach the same closed forms
    for blk in (1, 2, 3, len(x) + 1):
        outs.append(oracle.online_softmax_row(x, blk)[0])
        outs.append(oracle.split_softmax_row(x, blk)[0])
    for got in outs:
        for g, w in zip(got, want):
            if w == 0.0:
                assert g == 0.0
            else:
                assert abs(g - w) <= rtol * abs(w)


def test_softmax_brute_force_tiny(oracle):
    """3x5 random rows against 60-digit Decimal arithmetic: catches any
    wrong term, sign or index in the definition."""
    rng = _rng(11)
    x = rng.normal(0.0, 3.0, size=(3, 5))
    for row in x:
        got = oracle.softmax_row(row)
        want = bf_softmax(row)
        np.testing.assert_allclose(got, want, rtol=1e-14, atol=0)


@pytest.mark.parametrize("n", [1, 2, 5, 768, 4097])
def test_softmax_rows_sum_to_one_and_shift_invariant(oracle, n):
    """sum_j y_j = 1 and softmax(x + c) = softmax(x) for c = 7, 100, 1000.
    c = 1000 overflows exp() if the row maximum is not subtracted."""
    rng = _rng(n)
    x = rng.normal(0.0, 2.0, size=n)
    y = oracle.softmax_row(x)
    assert abs(math.fsum(y) - 1.0) <= 1e-13
    assert np.all(y > 0)
    for c in (7.0, 100.0, 1000.0):
        ys = oracle.softmax_row(x + c)
        np.testing.assert_allclose(ys, y, rtol=1e-12 * max(1.0, c / 10), atol=0)


def test_softmax_matches_torch_double(oracle):
    """Special case reducing to a library routine: torch.softmax in float64."""
    rng = _rng(3)
    x = rng.normal(0.0, 4.0, size=(17, 333))
    x[:, 100:] = np.where(rng.random((17, 233)) < 0.3, -np.inf, x[:, 100:])
    want = torch.softmax(torch.from_numpy(x), dim=-1).numpy()
    got = np.stack([oracle.softmax_row(r) for r in x])
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-300)
    assert np.all(got[np.isneginf(x)] == 0.0)


def test_softmax_nan_propagates_through_row(oracle):
    x = [0.0, 1.0, float("nan"), 2.0]
    assert np.all(np.isnan(oracle.softmax_row(x)))


def test_softmax_rows_batch_respects_ld_and_padding(oracle):
    """Batch form with ld > N and NaN padding: catches a stride / padding
    mistake (reading past N would turn rows into NaN)."""
    rng = _rng(5)
    M, N, ld = 6, 37, 48
    store = np.full((M, ld), np.nan, dtype=np.float32)
    store[:, :N] = rng.normal(0, 1, size=(M, N)).astype(np.float32)
    got = oracle.softmax(store[:, :N])
    assert np.all(np.isfinite(got))
    for r in range(M):
        np.testing.assert_array_equal(got[r], oracle.softmax_row(store[r, :N].astype(np.float64)))


# ----------------------------------------------------------------------------
# online / split-row softmax
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("block", [1, 2, 7, 64, 1000, 4096, 5000])
def test_online_and_split_agree_with_two_pass(oracle, block):
    """The (m, d) recurrence and the chunk-partial merge reach the direct
    definition (to 1e-14), and the final state is (max x, sum exp(x - max))
    computed exactly: catches a wrong rescale factor exp(m_old - m_new)
    (e.g. a flipped sign) or a dropped partial."""
    rng = _rng(block)
    x = rng.normal(0.0, 3.0, size=4096)
    x[rng.random(4096) < 0.01] += 25.0
    y_ref = oracle.softmax_row(x)
    m_exact = max(x)
    d_exact = float(sum((CTX.exp(_dec(v) - _dec(m_exact)) for v in x), Decimal(0)))
    for fn in (oracle.online_softmax_row, oracle.split_softmax_row):
        y, m, d = fn(x, block)
        np.testing.assert_allclose(y, y_ref, rtol=1e-13, atol=0)
        assert m == m_exact
        assert abs(d - d_exact) <= 1e-13 * d_exact


def test_online_state_after_each_block_is_prefix_softmax_state(oracle):
    """After any prefix of blocks the running state equals (max, sum exp(x -
    max)) of that prefix: pins the recurrence step by step, not just its end."""
    rng = _rng(21)
    x = rng.normal(0, 5, size=40)
    for k in range(1, 41):
        _, m, d = oracle.online_softmax_row(x[:k], 6)
        mk = max(x[:k])
        dk = float(sum((CTX.exp(_dec(v) - _dec(mk)) for v in x[:k]), Decimal(0)))
        assert m == mk
        assert abs(d - dk) <= 1e-14 * dk


def test_split_skips_fully_masked_chunks(oracle):
    """A chunk whose entries are all -inf has d_c = 0 and must be skipped, not
    merged through exp(-inf - (-inf)) = NaN."""
    x = np.full(64, -np.inf)
    x[40:48] = np.log(np.arange(1, 9))
    for chunk in (8, 16, 5):
        for fn in (oracle.split_softmax_row, oracle.online_softmax_row):
            y, m, d = fn(x, chunk)
            assert np.all(np.isfinite(y))
            np.testing.assert_allclose(y[40:48], np.arange(1, 9) / 36.0, rtol=1e-14)
            assert np.all(y[:40] == 0) and np.all(y[48:] == 0)
            assert m == np.log(8.0)


def test_split_all_masked_row_is_zero(oracle):
    y, m, d = oracle.split_softmax_row(np.full(10, -np.inf), 3)
    assert np.all(y == 0) and d == 0.0 and m == -np.inf


def test_outlier_rows_closed_form(oracle):
    """Rows like the online-softmax workload (N(0,1) with entries set to +30):
    each outlier gets 1 / (k + S) with S = sum over the rest of exp(x - 30),
    summed here with math.fsum."""
    rng = _rng(8)
    n = 1 << 14
    x = rng.normal(0, 1, size=n)
    hit = rng.random(n) < 1e-3
    x[hit] = 30.0
    k = int(hit.sum())
    assert k > 0
    S = math.fsum(math.exp(v - 30.0) for v in x[~hit])
    want = 1.0 / (k + S)
    for chunk in (1 << 10, 1 << 12, n):
        y, _, _ = oracle.split_softmax_row(x, chunk)
        np.testing.assert_allclose(y[hit], want, rtol=1e-13)
    y = oracle.split_softmax(x[None, :].astype(np.float32), 1 << 11)
    assert abs(math.fsum(y[0]) - 1.0) < 1e-12


# ----------------------------------------------------------------------------
# GELU
# ----------------------------------------------------------------------------
def test_gelu_constants_match_pages(oracle):
    c = _golden.read_constants("gelu_constants.txt")
    assert oracle.gelu_sqrt_2_over_pi() == float(c["gelu_sqrt_2_over_pi"])
    assert oracle.gelu_cubic() == float(c["gelu_cubic"])
    # the two printed forms of sqrt(2/pi) agree with the closed form
    assert abs(float(c["gelu_sqrt_2_over_pi"]) - math.sqrt(2 / math.pi)) < 1e-8
    assert abs(float(c["gelu_sqrt_2_over_pi_long"]) - math.sqrt(2 / math.pi)) < 1e-15
    assert float(c["layernorm_eps_default"]) == 1e-5


def test_gelu_special_values(oracle):
    """GELU(0) = 0; GELU(x) = x exactly once tanh rounds to 1 in double, which
    for u = 0.79788456 (x + 0.044715 x^3) > 19.1 holds from x = 8 on; GELU(x)
    is in [-1e-30, 0] for x <= -10."""
    assert oracle.gelu_tanh(0.0) == 0.0
    for x in (8.0, 9.5, 10.0, 50.0, 1e3, 3.0e10):
        assert oracle.gelu_tanh(x) == x
    for x in (-10.0, -13.0, -100.0, -1e4):
        g = oracle.gelu_tanh(x)
        assert -1e-30 <= g <= 0.0


def test_gelu_odd_identity(oracle):
    """tanh is odd, so GELU(x) - GELU(-x) = x exactly in real arithmetic:
    catches a sign error or a dropped 0.5 / '1 +' term."""
    for x in np.linspace(-12, 12, 97):
        assert abs(oracle.gelu_tanh(x) - oracle.gelu_tanh(-x) - x) <= 4e-16 * max(1.0, abs(x))


def test_gelu_brute_force(oracle):
    """Decimal (60 digits) evaluation of 0.5 z (1 + tanh(0.79788456 (z + 0.044715 z^3)))."""
    for z in (-6.0, -3.5, -2.0, -1.0, -0.25, 1e-6, 0.3, 1.0, 2.5, 5.0, 7.0):
        want = bf_gelu(z)
        # the double evaluation of 1 + tanh(u) loses digits for negative z
        tol = 1e-15 * max(1.0, abs(z)) + 4e-16 * abs(want)
        assert abs(oracle.gelu_tanh(z) - want) <= tol, z


def test_gelu_matches_torch_tanh_gelu(oracle):
    """torch's tanh-approximation GELU in float64 uses sqrt(2/pi) to full
    precision; against the printed 0.79788456 the gap is < 1e-9 relative."""
    z = np.linspace(-9, 9, 1001)
    want = torch.nn.functional.gelu(torch.from_numpy(z), approximate="tanh").numpy()
    got = oracle.gelu_tanh(z)
    np.testing.assert_allclose(got, want, rtol=0, atol=2e-9)


# ----------------------------------------------------------------------------
# LayerNorm, LayerNorm -> GELU
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("case", _golden.read_cases("layernorm_closed_forms.txt"), ids=lambda c: c[0])
def test_layernorm_golden_closed_forms(oracle, case):
    """Worked examples: catches an unbiased (n-1) variance, eps outside the
    sqrt, a wrong affine order and shift sensitivity."""
    _, params, rows = case
    x = [float(v) for v in rows["x"]]
    n = len(x)
    eps = float(params.get("eps", Decimal("1e-5")))
    w = [float(params["w"])] * n if "w" in params else None
    b = [float(params["b"])] * n if "b" in params else None
    want = [float(v) for v in rows["z"]]
    got = oracle.layernorm_row(x, w, b, eps)
    np.testing.assert_allclose(got, want, rtol=0, atol=2e-15 * max(1.0, max(abs(v) for v in want)))


def test_layernorm_unit_affine_moments(oracle):
    """With w = 1, b = 0: mean(z) = 0 and var(z) = s^2 / (s^2 + eps), where
    s^2 is the biased sample variance (numpy.var) of the row."""
    rng = _rng(7)
    for n in (5, 127, 768, 4097, 8192):
        x = rng.normal(0.3, 1.7, size=n)
        z = oracle.layernorm_row(x, None, None, 1e-5)
        s2 = float(np.var(x))
        assert abs(np.mean(z)) < 1e-13
        assert abs(np.mean(z * z) - s2 / (s2 + 1e-5)) < 1e-12


def test_layernorm_shift_invariant(oracle):
    rng = _rng(9)
    x = rng.normal(0, 1, size=300)
    w = rng.uniform(0.5, 1.5, size=300)
    b = rng.normal(0, 0.1, size=300)
    z0 = oracle.layernorm_row(x, w, b, 1e-5)
    z1 = oracle.layernorm_row(x + 1000.0, w, b, 1e-5)
    np.testing.assert_allclose(z1, z0, rtol=0, atol=5e-11)


def test_layernorm_brute_force_with_affine(oracle):
    rng = _rng(13)
    x = rng.normal(0, 2, size=(3, 5))
    w = rng.uniform(0.5, 1.5, size=5)
    b = rng.normal(0, 0.1, size=5)
    for row in x:
        want = [float(v) for v in bf_layernorm(row, w, b, 1e-5)]
        np.testing.assert_allclose(oracle.layernorm_row(row, w, b, 1e-5), want, rtol=0, atol=1e-15)
        want_g = [bf_gelu(v) for v in want]
        np.testing.assert_allclose(oracle.layernorm_gelu_row(row, w, b, 1e-5), want_g, rtol=0, atol=4e-15)


def test_layernorm_matches_torch_double(oracle):
    rng = _rng(17)
    M, N = 9, 769
    x = rng.normal(0, 1, size=(M, N)).astype(np.float32)
    w = rng.uniform(0.5, 1.5, size=N).astype(np.float32)
    b = rng.normal(0, 0.1, size=N).astype(np.float32)
    xt, wt, bt = (torch.from_numpy(a).double() for a in (x, w, b))
    z_t = torch.nn.functional.layer_norm(xt, (N,), wt, bt, 1e-5)
    np.testing.assert_allclose(oracle.layernorm(x, w, b, 1e-5), z_t.numpy(), rtol=0, atol=1e-13)
    g_t = torch.nn.functional.gelu(z_t, approximate="tanh")
    np.testing.assert_allclose(oracle.layernorm_gelu(x, w, b, 1e-5), g_t.numpy(), rtol=0, atol=5e-9)


def test_layernorm_gelu_is_gelu_of_layernorm(oracle):
    """The fused form applies GELU after the affine step (not before it, not
    to the normalised value without w, b)."""
    rng = _rng(19)
    x = rng.normal(0, 1, size=(4, 50)).astype(np.float32)
    w = rng.uniform(0.5, 1.5, size=50).astype(np.float32)
    b = rng.normal(0, 0.5, size=50).astype(np.float32)
    z = oracle.layernorm(x, w, b, 1e-5)
    g = oracle.layernorm_gelu(x, w, b, 1e-5)
    np.testing.assert_array_equal(g, oracle.gelu_tanh(z))


def test_layernorm_rows_batch_respects_ld_and_null_affine(oracle):
    """Batch form: ld > N with NaN padding never reaches the statistics; a
    NULL weight / bias means 1 / 0."""
    rng = _rng(23)
    M, N, ld = 5, 127, 136
    store = np.full((M, ld), np.nan, dtype=np.float32)
    store[:, :N] = rng.normal(0, 1, size=(M, N)).astype(np.float32)
    g = oracle.layernorm_gelu(store[:, :N], None, None, 1e-5)
    assert np.all(np.isfinite(g))
    ones, zeros = np.ones(N, np.float32), np.zeros(N, np.float32)
    np.testing.assert_array_equal(g, oracle.layernorm_gelu(np.ascontiguousarray(store[:, :N]), ones, zeros, 1e-5))
    for r in range(M):
        np.testing.assert_array_equal(g[r], oracle.layernorm_gelu_row(store[r, :N].astype(np.float64), None, None, 1e-5))


# ----------------------------------------------------------------------------
# RMSNorm, fused residual + RMSNorm
# ----------------------------------------------------------------------------
def bf_rmsnorm(xs, w=None, eps=1e-5):
    xd = [_dec(v) for v in xs]
    ms = CTX.divide(sum((v * v for v in xd), Decimal(0)), len(xd))
    inv = CTX.divide(1, CTX.sqrt(ms + _dec(eps)))
    return [float(CTX.multiply(CTX.multiply(v, inv), _dec(w[j]) if w is not None else Decimal(1)))
            for j, v in enumerate(xd)]


@pytest.mark.parametrize("case", _golden.read_cases("rmsnorm_closed_forms.txt"), ids=lambda c: c[0])
def test_rmsnorm_golden_closed_forms(oracle, case):
    """Worked examples: catches a subtracted mean, an (n-1) or missing 1/n,
    eps outside the sqrt, a dropped weight and a residual that is not added."""
    _, params, rows = case
    x = [float(v) for v in rows["x"]]
    eps = float(params.get("eps", Decimal("1e-5")))
    w = [float(v) for v in rows["w"]] if "w" in rows else None
    want = [float(v) for v in rows["y"]]
    tol = 2e-15 * max(1.0, max(abs(v) for v in want))
    if "r" in rows:
        r = [float(v) for v in rows["r"]]
        s, got = oracle.residual_rmsnorm_row(x, r, w, eps, "exact")
        np.testing.assert_array_equal(s, [float(v) for v in rows["s"]])
    else:
        got = oracle.rmsnorm_row(x, w, eps)
    np.testing.assert_allclose(got, want, rtol=0, atol=tol)


def test_rmsnorm_unit_weight_moments_scale_and_sign(oracle):
    """With w = 1: mean(y^2) = ms / (ms + eps) (ms = mean(x^2), from numpy);
    with eps = 0, y is unchanged by scaling the row and odd in x; unlike
    LayerNorm, shifting the row changes y."""
    rng = _rng(29)
    for n in (5, 127, 768, 4097, 8192):
        x = rng.normal(0.3, 1.7, size=n)
        ms = float(np.mean(x * x))
        y = oracle.rmsnorm_row(x, None, 1e-5)
        assert abs(np.mean(y * y) - ms / (ms + 1e-5)) < 1e-12
        y0 = oracle.rmsnorm_row(x, None, 0.0)
        np.testing.assert_allclose(oracle.rmsnorm_row(7.0 * x, None, 0.0), y0, rtol=0, atol=1e-14)
        np.testing.assert_array_equal(oracle.rmsnorm_row(-x, None, 0.0), -y0)
        assert np.max(np.abs(oracle.rmsnorm_row(x + 1.0, None, 0.0) - y0)) > 1e-3


def test_rmsnorm_brute_force_with_weight(oracle):
    rng = _rng(31)
    x = rng.normal(0, 2, size=(3, 5))
    w = rng.uniform(0.5, 1.5, size=5)
    for row in x:
        np.testing.assert_allclose(oracle.rmsnorm_row(row, w, 1e-5), bf_rmsnorm(row, w, 1e-5), rtol=0, atol=1e-15)


def test_rmsnorm_matches_torch_double(oracle):
    rng = _rng(37)
    M, N = 9, 769
    x = rng.normal(0, 1, size=(M, N)).astype(np.float32)
    w = rng.uniform(0.5, 1.5, size=N).astype(np.float32)
    xt, wt = torch.from_numpy(x).double(), torch.from_numpy(w).double()
    y_t = torch.nn.functional.rms_norm(xt, (N,), wt, 1e-5)
    np.testing.assert_allclose(oracle.rmsnorm(x, w, 1e-5), y_t.numpy(), rtol=0, atol=1e-13)


def test_round_to_storage_types(oracle):
    """bf16: the same value as torch's float32 -> bfloat16 conversion (round
    to nearest even) on fp32 inputs, including exact ties; f32: numpy's
    float64 -> float32 conversion."""
    rng = _rng(41)
    v32 = (rng.normal(0, 3, size=2000) * np.exp2(rng.integers(-20, 20, size=2000))).astype(np.float32)
    want = torch.from_numpy(v32).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(oracle.round_to(v32.astype(np.float64), "bf16"), want)
    ties = np.array([1 + 2.0**-8, 1 + 3 * 2.0**-8, -(1 + 2.0**-8), 2 + 2.0**-7, 1 + 2.0**-8 + 2.0**-20])
    np.testing.assert_array_equal(oracle.round_to(ties, "bf16"), [1.0, 1 + 2.0**-6, -1.0, 2.0, 1 + 2.0**-7])
    v64 = rng.normal(0, 5, size=2000)
    np.testing.assert_array_equal(oracle.round_to(v64, "f32"), v64.astype(np.float32).astype(np.float64))
    np.testing.assert_array_equal(oracle.round_to(v64, "exact"), v64)


@pytest.mark.parametrize("storage,dt", [("bf16", torch.bfloat16), ("f32", torch.float32)])
def test_residual_rmsnorm_is_rmsnorm_of_stored_sum(oracle, storage, dt):
    """residual_out is x + residual as the storage type holds it (torch's own
    addition in that dtype), and out is the RMSNorm of that stored tensor, not
    of the unrounded sum."""
    rng = _rng(43)
    M, N = 6, 513
    x = torch.from_numpy(rng.normal(0, 1, size=(M, N)).astype(np.float32)).to(dt)
    r = torch.from_numpy(rng.normal(0, 1, size=(M, N)).astype(np.float32)).to(dt)
    w = torch.from_numpy(rng.uniform(0.5, 1.5, size=N).astype(np.float32)).to(dt)
    s_t = x + r
    s, y = oracle.residual_rmsnorm(x.float().numpy(), r.float().numpy(), w.float().numpy(), 1e-5, storage)
    np.testing.assert_array_equal(s, s_t.double().numpy())
    y_t = torch.nn.functional.rms_norm(s_t.double(), (N,), w.double(), 1e-5)
    np.testing.assert_allclose(y, y_t.numpy(), rtol=0, atol=1e-13)
    if storage == "bf16":  # the norm of the unrounded sum differs visibly
        y_exact = oracle.rmsnorm((x.double() + r.double()).float().numpy(), w.float().numpy(), 1e-5)
        assert np.max(np.abs(y_exact - y)) > 1e-4


def test_rmsnorm_rows_batch_respects_ld_and_null_weight(oracle):
    rng = _rng(47)
    M, N, ld = 5, 127, 136
    store = np.full((M, ld), np.nan, dtype=np.float32)
    store[:, :N] = rng.normal(0, 1, size=(M, N)).astype(np.float32)
    y = oracle.rmsnorm(store[:, :N], None, 1e-5)
    assert np.all(np.isfinite(y))
    np.testing.assert_array_equal(y, oracle.rmsnorm(np.ascontiguousarray(store[:, :N]), np.ones(N, np.float32), 1e-5))
    for i in range(M):
        np.testing.assert_array_equal(y[i], oracle.rmsnorm_row(store[i, :N].astype(np.float64), None, 1e-5))
    # the residual form with both inputs padded to the same stride
    rstore = np.full((M, ld), np.nan, dtype=np.float32)
    rstore[:, :N] = rng.normal(0, 1, size=(M, N)).astype(np.float32)
    s, yr = oracle.residual_rmsnorm(store[:, :N], rstore[:, :N], None, 1e-5, "f32")
    assert np.all(np.isfinite(s)) and np.all(np.isfinite(yr))
    for i in range(M):
        si, yi = oracle.residual_rmsnorm_row(store[i, :N], rstore[i, :N], None, 1e-5, "f32")
        np.testing.assert_array_equal(s[i], si)
        np.testing.assert_array_equal(yr[i], yi)


# ----------------------------------------------------------------------------
# causal softmax
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("case", _golden.read_cases("softmax_causal_closed_forms.txt"), ids=lambda c: c[0])
def test_softmax_causal_golden_closed_forms(oracle, case):
    """Worked examples: catches a kept count off by one, a mask that ignores
    the period or the offset, and masked entries that are read."""
    _, params, rows = case
    r, period, offset = int(params["r"]), int(params["period"]), int(params["offset"])
    x = [float(v) for v in rows["x"]]
    want = [float(v) for v in rows["y"]]
    got = oracle.softmax_causal_rows_at(x, r, period, offset)
    np.testing.assert_allclose(got, want, rtol=0, atol=2e-16)
    # the batch form at the same row index
    M = r + 1
    xb = np.zeros((M, len(x)), np.float32)
    xb[r] = np.float32(x)
    np.testing.assert_allclose(oracle.softmax_causal(xb, period, offset)[r], want, rtol=0, atol=1e-7)


def test_causal_kept_count(oracle):
    """kept = clamp(r mod period + offset + 1, 0, n), against a count of the
    columns c with c <= r mod period + offset."""
    for n in (1, 5, 64):
        for period in (1, 3, 64, 100):
            for offset in (-70, -3, -1, 0, 2, 63, 1000):
                for r in (0, 1, 2, 63, 64, 99, 12345):
                    want = sum(1 for c in range(n) if c <= r % period + offset)
                    assert oracle.causal_kept(r, n, period, offset) == want


def test_softmax_causal_matches_torch_on_masked_input(oracle):
    """Equals torch's softmax of the row with the masked columns set to -inf
    (zeros where torch's all -inf row gives NaN), whatever the masked columns
    hold: here NaN and +inf, which any read would propagate."""
    rng = _rng(53)
    M, N, period, offset = 37, 40, 16, 3
    x = rng.normal(0, 3, size=(M, N)).astype(np.float32)
    xm = x.copy()
    for r in range(M):
        keep = r % period + offset
        xm[r, keep + 1:] = -np.inf
        x[r, keep + 1:] = np.nan if r % 2 else np.inf
    want = torch.softmax(torch.from_numpy(xm).double(), dim=1).numpy()
    got = oracle.softmax_causal(x, period, offset)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)


def test_softmax_causal_degenerate_masks(oracle):
    rng = _rng(59)
    x = rng.normal(0, 1, size=(9, 33)).astype(np.float32)
    # a mask that keeps everything is the plain softmax; one that keeps nothing is all zeros
    np.testing.assert_allclose(oracle.softmax_causal(x, 1, 33), torch.softmax(torch.from_numpy(x).double(), 1).numpy(),
                               rtol=0, atol=1e-15)
    assert np.all(oracle.softmax_causal(x, 4, -5) == 0.0)


# ----------------------------------------------------------------------------
# exact GELU, row sum, row max
# ----------------------------------------------------------------------------
_GR = {c[0]: c for c in _golden.read_cases("gelu_erf_and_row_reductions.txt")}


def test_gelu_erf_table_values(oracle):
    """x * Phi(x) at printed standard normal CDF values: catches a missing
    1/sqrt(2), the tanh approximation in its place, or a dropped 0.5."""
    _, _, rows = _GR["gelu_table"]
    z = [float(v) for v in rows["z"]]
    want = [float(v) for v in rows["g"]]
    np.testing.assert_allclose(oracle.gelu_erf(z), want, rtol=0, atol=4e-16)


def test_gelu_erf_identities_and_libraries(oracle):
    """GELU(x) - GELU(-x) = x; equal to x * scipy.special.ndtr(x) and torch's
    exact GELU in float64; within the known ~5e-4 of the tanh form."""
    sp = pytest.importorskip("scipy.special")
    z = np.linspace(-12, 12, 2401)
    g = oracle.gelu_erf(z)
    np.testing.assert_allclose(g - oracle.gelu_erf(-z), z, rtol=0, atol=4e-15)
    np.testing.assert_allclose(g, z * sp.ndtr(z), rtol=1e-13, atol=1e-300)  # relative, tail included
    # torch evaluates 1 + erf itself, which cancels in the negative tail: absolute
    g_t = torch.nn.functional.gelu(torch.from_numpy(z), approximate="none").numpy()
    np.testing.assert_allclose(g, g_t, rtol=2e-15, atol=2e-15)
    assert np.max(np.abs(g - oracle.gelu_tanh(z))) < 5e-4
    assert np.max(np.abs(g - oracle.gelu_tanh(z))) > 1e-4  # and it is the other function


def test_layernorm_gelu_erf_is_erf_gelu_of_layernorm(oracle):
    rng = _rng(61)
    x = rng.normal(0, 1, size=(5, 300)).astype(np.float32)
    w = rng.uniform(0.5, 1.5, size=300).astype(np.float32)
    b = rng.normal(0, 0.1, size=300).astype(np.float32)
    np.testing.assert_array_equal(oracle.layernorm_gelu_erf(x, w, b, 1e-5), oracle.gelu_erf(oracle.layernorm(x, w, b, 1e-5)))
    ref = torch.nn.functional.gelu(torch.nn.functional.layer_norm(torch.from_numpy(x).double(), (300,),
                                   torch.from_numpy(w).double(), torch.from_numpy(b).double(), 1e-5),
                                   approximate="none").numpy()
    np.testing.assert_allclose(oracle.layernorm_gelu_erf(x, w, b, 1e-5), ref, rtol=0, atol=1e-13)


@pytest.mark.parametrize("name", ["ramp", "cancelling", "negative_with_padding_values", "single"])
def test_row_sum_and_max_worked_examples(oracle, name):
    _, _, rows = _GR[name]
    x = np.array([[float(v) for v in rows["x"]]], dtype=np.float32)
    assert oracle.row_sum(x)[0] == float(rows["sum"][0])
    assert oracle.row_max(x)[0] == float(rows["max"][0])


def test_row_sum_matches_exactly_rounded_sum(oracle):
    """Against math.fsum (an exactly rounded sum, a different algorithm): the
    double left-to-right sum of fp32 inputs is within N * 2^-53 * sum|x|;
    also sum(x + c) = sum(x) + N c."""
    import math

    rng = _rng(67)
    for n in (1, 7, 768, 4097, 100003):
        x = rng.normal(0, 3, size=(3, n)).astype(np.float32)
        got = oracle.row_sum(x)
        for i in range(3):
            want = math.fsum(float(v) for v in x[i])
            assert abs(got[i] - want) <= n * 2.0**-53 * float(np.abs(x[i]).astype(np.float64).sum())
    # integer-valued rows: every partial sum is exact, so the result is too
    xi = rng.integers(-1000, 1000, size=(4, 100003)).astype(np.float32)
    np.testing.assert_array_equal(oracle.row_sum(xi), xi.astype(np.int64).sum(axis=1).astype(np.float64))


def test_row_max_special_rows(oracle):
    """Matches numpy's max on ordinary rows; a NaN anywhere makes NaN; an all
    -inf row gives -inf; the stride's padding is never read."""
    rng = _rng(71)
    M, N, ld = 6, 129, 140
    store = np.full((M, ld), np.nan, dtype=np.float32)
    store[:, :N] = rng.normal(0, 1, size=(M, N)).astype(np.float32)
    store[1, :N] = -np.inf
    store[2, 77] = np.nan
    store[3, 5] = np.inf
    out = oracle.row_max(store[:, :N])
    want = store[:, :N].astype(np.float64).max(axis=1)
    np.testing.assert_array_equal(out, want)  # numpy's max propagates NaN too
    assert out[1] == -np.inf and np.isnan(out[2]) and out[3] == np.inf
    s = oracle.row_sum(store[:, :N])
    assert s[1] == -np.inf and np.isnan(s[2]) and s[3] == np.inf and np.all(np.isfinite(s[[0, 4, 5]]))


# ----------------------------------------------------------------------------
# LayerNorm -> affine -> tanh-GELU backward
# ----------------------------------------------------------------------------
def test_gelu_tanh_grad_values(oracle):
    """g'(0) = 1/2 exactly; g' -> 1 and -> 0 in the tails; the derivative of
    the oracle's own GELU by central differences."""
    assert oracle.gelu_tanh_grad(0.0) == 0.5
    assert abs(oracle.gelu_tanh_grad(12.0) - 1.0) < 1e-15 and abs(oracle.gelu_tanh_grad(-12.0)) < 1e-15
    z = np.linspace(-6, 6, 241)
    h = 1e-5
    fd = (oracle.gelu_tanh(z + h) - oracle.gelu_tanh(z - h)) / (2 * h)
    np.testing.assert_allclose(oracle.gelu_tanh_grad(z), fd, rtol=0, atol=1e-9)


def test_layernorm_gelu_backward_matches_torch_autograd(oracle):
    """torch's float64 autograd through gelu(layer_norm(x), approximate="tanh")
    (which uses sqrt(2/pi) for 0.79788456: a 1e-9 relative difference)."""
    rng = _rng(73)
    M, N = 7, 129
    x = rng.normal(0.5, 1.5, size=(M, N)).astype(np.float32)
    dy = rng.normal(0, 1, size=(M, N)).astype(np.float32)
    w = rng.uniform(0.5, 1.5, size=N).astype(np.float32)
    b = rng.normal(0, 0.1, size=N).astype(np.float32)
    dx, dw, db = oracle.layernorm_gelu_backward(x, dy, w, b, 1e-5)
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    wt = torch.tensor(w, dtype=torch.float64, requires_grad=True)
    bt = torch.tensor(b, dtype=torch.float64, requires_grad=True)
    y = torch.nn.functional.gelu(torch.nn.functional.layer_norm(xt, (N,), wt, bt, 1e-5), approximate="tanh")
    y.backward(torch.tensor(dy, dtype=torch.float64))
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=0, atol=1e-8)
    np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=0, atol=1e-8)
    np.testing.assert_allclose(db, bt.grad.numpy(), rtol=0, atol=1e-8)


def test_layernorm_gelu_backward_central_differences(oracle):
    """Each gradient entry against (L(p + h) - L(p - h)) / 2h of L = sum dy * y
    with the oracle's own forward: catches a dropped GELU derivative, a dropped
    mean or variance term, or dw / db from the wrong factor."""
    rng = _rng(79)
    n = 9
    x = rng.normal(0.3, 1.2, size=n)
    dy = rng.normal(0, 1, size=n)
    w = rng.uniform(0.5, 1.5, size=n)
    b = rng.normal(0, 0.3, size=n)
    dx, dw, db = oracle.layernorm_gelu_backward_row(x, dy, w, b, 1e-3)
    loss = lambda xx, ww, bb: float(np.dot(dy, oracle.layernorm_gelu_row(xx, ww, bb, 1e-3)))
    h = 1e-6
    for j in range(n):
        e = np.zeros(n)
        e[j] = h
        assert abs((loss(x + e, w, b) - loss(x - e, w, b)) / (2 * h) - dx[j]) < 1e-7
        assert abs((loss(x, w + e, b) - loss(x, w - e, b)) / (2 * h) - dw[j]) < 1e-7
        assert abs((loss(x, w, b + e) - loss(x, w, b - e)) / (2 * h) - db[j]) < 1e-7


def test_layernorm_gelu_backward_projections(oracle):
    """The normalised row ignores a shift of x: sum_j dx_j = 0; with eps = 0 it
    also ignores a scale: sum_j dx_j xh_j = 0."""
    rng = _rng(83)
    for n in (5, 768, 4097):
        x = rng.normal(1.0, 2.0, size=n)
        dy = rng.normal(0, 1, size=n)
        w = rng.uniform(0.5, 1.5, size=n)
        b = rng.normal(0, 0.1, size=n)
        dx, _, _ = oracle.layernorm_gelu_backward_row(x, dy, w, b, 1e-5)
        assert abs(dx.sum()) < 1e-12 * n
        dx0, _, _ = oracle.layernorm_gelu_backward_row(x, dy, w, b, 0.0)
        xh = (x - x.mean()) / x.std()
        assert abs(np.dot(dx0, xh)) < 1e-11 * n


def test_layernorm_gelu_backward_batch_respects_ld(oracle):
    """Batch form on rows padded with NaN to a stride ld > N (x and dy):
    equal to the row form; dw, db summed over the rows."""
    rng = _rng(89)
    M, N, ld = 4, 37, 45
    xs = np.full((M, ld), np.nan, dtype=np.float32)
    gs = np.full((M, ld), np.nan, dtype=np.float32)
    xs[:, :N] = rng.normal(0, 1, size=(M, N)).astype(np.float32)
    gs[:, :N] = rng.normal(0, 1, size=(M, N)).astype(np.float32)
    w = rng.uniform(0.5, 1.5, size=N).astype(np.float32)
    dx, dw, db = oracle.layernorm_gelu_backward(xs[:, :N], gs[:, :N], w, None, 1e-5)
    dw_sum, db_sum = np.zeros(N), np.zeros(N)
    for i in range(M):
        dxi, dwi, dbi = oracle.layernorm_gelu_backward_row(xs[i, :N], gs[i, :N], w, None, 1e-5)
        np.testing.assert_array_equal(dx[i], dxi)
        dw_sum += dwi
        db_sum += dbi
    np.testing.assert_allclose(dw, dw_sum, rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(db, db_sum, rtol=1e-15, atol=1e-15)


def test_batch_rejects_bad_shapes(oracle):
    with pytest.raises(ValueError):
        oracle.layernorm_gelu(np.zeros((2, 3), np.float32), np.ones(4, np.float32))


# ----------------------------------------------------------------------------
# fused residual + bias + GELU
# ----------------------------------------------------------------------------
def test_bias_residual_gelu_golden_closed_form(oracle):
    """Dyadic x, b, residual whose sums hit the exact-GELU table: catches a
    dropped bias or residual, a bias indexed by row, and the tanh form in
    place of the exact one."""
    (_, _, rows), = _golden.read_cases("bias_residual_gelu_closed_forms.txt")
    f = lambda k: np.array([float(v) for v in rows[k]], dtype=np.float64)
    x = np.stack([f("x0"), f("x1")]).astype(np.float32)
    r = np.stack([f("r0"), f("r1")]).astype(np.float32)
    b = f("b").astype(np.float32)
    want = np.stack([f("y0"), f("y1")])
    np.testing.assert_allclose(oracle.bias_residual_gelu(x, r, b), want, rtol=0, atol=4e-16)


@pytest.mark.parametrize("approximate", ["none", "tanh"])
def test_bias_residual_gelu_matches_torch(oracle, approximate):
    """torch's float64 GELU of x + b + residual on a non-square batch, with and
    without each of the optional inputs, both GELU forms."""
    rng = _rng(97)
    x = rng.normal(0, 2, size=(7, 13)).astype(np.float32)
    r = rng.normal(0, 1, size=(7, 13)).astype(np.float32)
    b = rng.normal(0, 0.5, size=13).astype(np.float32)
    g = lambda s: torch.nn.functional.gelu(torch.from_numpy(s), approximate=approximate).numpy()
    xd, rd, bd = x.astype(np.float64), r.astype(np.float64), b.astype(np.float64)
    # the tanh form: the pages' 0.79788456 against torch's sqrt(2 / pi), 1e-9 apart relatively
    atol = 1e-14 if approximate == "none" else 1e-9
    for res, bias, s in ((r, b, xd + bd + rd), (None, b, xd + bd), (r, None, xd + rd), (None, None, xd)):
        np.testing.assert_allclose(oracle.bias_residual_gelu(x, res, bias, approximate), g(s), rtol=0, atol=atol)


def test_bias_residual_gelu_strides(oracle):
    """x padded with NaN to a stride ld > N, the residual to another stride:
    equal to the contiguous computation."""
    rng = _rng(101)
    M, N = 5, 9
    x = rng.normal(size=(M, N)).astype(np.float32)
    r = rng.normal(size=(M, N)).astype(np.float32)
    b = rng.normal(size=N).astype(np.float32)
    xp = np.full((M, 12), np.nan, np.float32)
    xp[:, :N] = x
    rp = np.full((M, 16), np.nan, np.float32)
    rp[:, :N] = r
    want = oracle.bias_residual_gelu(x, r, b)
    np.testing.assert_array_equal(oracle.bias_residual_gelu(xp[:, :N], rp[:, :N], b), want)
    np.testing.assert_array_equal(oracle.bias_residual_gelu(xp[:, :N], r, b), want)
    rq = np.full((M, 12), np.nan, np.float32)  # the same padded stride as x: passed through as is
    rq[:, :N] = r
    np.testing.assert_array_equal(oracle.bias_residual_gelu(xp[:, :N], rq[:, :N], b), want)
