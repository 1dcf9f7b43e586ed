"""Coefficients of the exact-GELU evaluation used by the kernels.

The exact GELU is z * Phi(z), Phi the standard normal distribution function,
Phi(z) = 0.5 (1 + erf(z / sqrt 2)) ["Triton Kernel 实现练习" §3.4]. Its tanh
approximation ["CS336 Kernels, Triton" notes, "Triton GeLU"] is the same product
with Phi replaced by a logistic function of an odd cubic,
0.5 (1 + tanh(u)) = 1 / (1 + exp(-2u)), 2u = 1.5957691 z + 0.0713548 z^3.

The kernels keep that shape and raise the degree: Phi(z) ~ 1 / (1 + exp(-P(z)))
with P(z) = z (c0 + c1 z^2 + ... + c6 z^12), c fitted here so that the GELU's
absolute error z |sigma(P(z)) - Phi(z)| is as small as possible over |z| <= 8
(minimax on a dense grid, solved as a linear program in c after linearising:
the GELU error is z Phi (1 - Phi) |P - logit Phi| to first order). Beyond the
fitted range P must keep growing, so that sigma(P) tends to 1 (and to 0 for
z -> -inf) as Phi does: the program also asks P' >= 0 on [8, 60], and c6 >= 0.

Result: GELU error below 7e-8 over the fitted range; in fp32 the evaluation
adds its own rounding (tests/test_gelu_erf_form.py measures both). The cost is
one exp2 and one reciprocal per value, as in the tanh form, plus five more
fused multiply-adds, against an erfc rational approximation's two special
function calls and longer polynomial.

Run ``python -m row_wise_reduction_gb300.gelu_erf_fit`` to print the constants;
``csrc/ln_gelu_kernels.cuh`` holds the printed values. Needs numpy and scipy
(host only; the library does not import this module).
"""
from __future__ import annotations

import numpy as np

DEGREE = 6  # P(z) = z * sum_{k <= DEGREE} c_k z^{2k}
Z_FIT = 8.0
Z_MONOTONE = 60.0


def logit_phi(z: np.ndarray) -> np.ndarray:
    """log(Phi(z) / (1 - Phi(z))), without cancellation for large |z|."""
    from scipy.special import log_ndtr

    return log_ndtr(z) - log_ndtr(-z)


def fit(degree: int = DEGREE, z_fit: float = Z_FIT, z_mono: float = Z_MONOTONE, n: int = 6000):
    """Minimax coefficients c_0..c_degree and the linearised maximum GELU error."""
    from scipy.optimize import linprog
    from scipy.special import ndtr

    z = np.concatenate([np.linspace(1e-4, 3.0, n), np.linspace(3.0, z_fit, n // 2)])
    target = logit_phi(z)
    phi = ndtr(z)
    # d(GELU error) / d(P error), scaled by 1e6 so that the program's unknowns
    # and its error are far above the solver's feasibility tolerance (1e-7)
    weight = 1e6 * z * phi * (1.0 - phi)
    s = z / z_fit  # basis in s = z / z_fit: every column is at most 1
    basis = np.stack([s ** (2 * k + 1) for k in range(degree + 1)], axis=1)
    wb, wt = weight[:, None] * basis, weight * target
    ones = np.ones((len(z), 1))
    # unknowns b_0..b_degree (c_k = b_k / z_fit^(2k+1)) and e: minimise e with
    # -e <= w (basis b - target) <= e
    a_ub = [np.hstack([wb, -ones]), np.hstack([-wb, -ones])]
    b_ub = [wt, -wt]
    sg = np.linspace(1.0, z_mono / z_fit, 2000)
    slope = np.stack([(2 * k + 1) * sg ** (2 * k) for k in range(degree + 1)], axis=1)
    slope /= np.abs(slope).max(axis=1, keepdims=True)  # rows scaled to 1 (P' >= 0 only)
    a_ub.append(np.hstack([-slope, np.zeros((len(sg), 1))]))
    b_ub.append(np.zeros(len(sg)))
    bounds = [(None, None)] * degree + [(0.0, None), (0.0, None)]
    res = linprog(np.r_[np.zeros(degree + 1), 1.0], A_ub=np.vstack(a_ub), b_ub=np.concatenate(b_ub),
                  bounds=bounds, method="highs")
    if res.x is None:
        raise RuntimeError(f"linear program failed: {res.message}")
    c = res.x[:-1] / z_fit ** (2 * np.arange(degree + 1) + 1)
    return c, float(res.x[-1]) * 1e-6


def main() -> None:
    c, err = fit()
    print(f"// GELU error of the fit (linearised, |z| <= {Z_FIT}): {err:.3e}")
    for k, ck in enumerate(c):
        print(f"c{k} = {ck:.12e}")


if __name__ == "__main__":
    main()
