"""The kernels' evaluation of the exact GELU, checked on the CPU.

The kernels compute z Phi(z) ["Triton Kernel 实现练习" §3.4] as z / (1 + exp(-P(z)))
with an odd polynomial P whose coefficients csrc/ln_gelu_kernels.cuh holds
(struct GeluErfFit) and row_wise_reduction_gb300/gelu_erf_fit.py prints. These
tests read the constants from the header and check them against the
mathematics, with scipy's normal distribution function as the reference:
the error of the form itself, the limits, and an fp32 emulation of the kernels'
evaluation (correctly rounded exp2 and reciprocal standing in for the
approximate hardware ones, which the GPU parity tests cover)."""
import os
import re

import numpy as np
import pytest

scipy_special = pytest.importorskip("scipy.special")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "row_wise_reduction_gb300", "csrc", "ln_gelu_kernels.cuh")
LOG2E = 1.4426950408889634


@pytest.fixture(scope="module")
def coef():
    text = open(HEADER).read()
    block = text[text.index("struct GeluErfFit"):]
    block = block[:block.index("};")]
    c = {int(k): float(v) for k, v in re.findall(r"\bc(\d) = ([-+0-9.e]+)", block)}
    assert sorted(c) == list(range(7))
    return np.array([c[k] for k in range(7)])


def P(c, z):
    return z * sum(ck * z ** (2 * k) for k, ck in enumerate(c))


def gelu(z):
    return z * scipy_special.ndtr(z)


def test_form_error_within_7e8(coef):
    z = np.linspace(-16.0, 16.0, 1_600_001)
    with np.errstate(over="ignore"):
        approx = z / (1.0 + np.exp(-P(coef, z)))
    assert np.max(np.abs(approx - gelu(z))) < 7e-8


def test_polynomial_increasing_and_odd(coef):
    z = np.linspace(0.0, 200.0, 400_001)
    dp = sum((2 * k + 1) * ck * z ** (2 * k) for k, ck in enumerate(coef))
    assert np.all(dp > 0)
    assert coef[-1] > 0  # P -> +inf as z -> +inf (and -inf as z -> -inf)
    np.testing.assert_allclose(P(coef, -z), -P(coef, z), rtol=1e-14, atol=0)


def test_slope_at_zero_is_that_of_logit_phi(coef):
    # logit(Phi(z)) = 4 z / sqrt(2 pi) + O(z^3): the fit keeps Phi'(0) = 1 / sqrt(2 pi)
    assert abs(coef[0] - 4.0 / np.sqrt(2.0 * np.pi)) < 1e-5


def test_fit_script_reproduces_the_header(coef):
    pytest.importorskip("scipy.optimize")
    from row_wise_reduction_gb300 import gelu_erf_fit

    c, err = gelu_erf_fit.fit()
    assert err < 7e-8
    z = np.linspace(-10.0, 10.0, 200_001)
    with np.errstate(over="ignore"):
        a = z / (1.0 + np.exp(-P(c, z)))
        b = z / (1.0 + np.exp(-P(coef, z)))
    assert np.max(np.abs(a - b)) < 1e-9


def emulate_f32(coef, z):
    """The kernels' operations in fp32, one rounding per operation."""
    f = np.float32
    z = z.astype(f)
    q = [f(-LOG2E * ck) for ck in coef]
    with np.errstate(over="ignore", invalid="ignore"):
        z2 = z * z
        acc = np.full_like(z, q[6])
        for k in range(5, -1, -1):
            acc = (acc.astype(np.float64) * z2 + np.float64(q[k])).astype(f)  # one rounding: fma
        a = acc * z
        e = np.exp2(a.astype(np.float64)).astype(f)
        d = e + f(1.0)
        r = (1.0 / d.astype(np.float64)).astype(f)
        return z * r


def test_fp32_evaluation_error(coef):
    z = np.concatenate([np.linspace(-12.0, 12.0, 400_001), np.array([0.0, -0.0, 1e-30, -1e-30, 30.0, -30.0])])
    got = emulate_f32(coef, z).astype(np.float64)
    zf = z.astype(np.float32).astype(np.float64)
    ref = gelu(zf)
    # rounding of the exp2 argument a = -log2(e) P(z), |a| <= |z| (2.31 + 0.105 z^2) for |z| <= 12,
    # becomes ~|a| 2^-24 relative error of the result; plus the form's 7e-8
    arg = np.abs(zf) * (2.31 + 0.105 * zf**2)
    bound = (1.0 + arg) * 2e-7 * np.abs(ref) + 7e-8 + 1e-37
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) - bound))


def test_fp32_limits(coef):
    z = np.array([1e3, 1e6, 3e38, np.inf, -1e3, -1e6, -3e38, np.nan], dtype=np.float32)
    got = emulate_f32(coef, z)
    np.testing.assert_array_equal(got[:4], z[:4])  # z for large positive z
    assert np.all(got[4:7] == 0.0) and np.all(np.signbit(got[4:7]))  # -0 for large negative z
    assert np.isnan(got[7])
