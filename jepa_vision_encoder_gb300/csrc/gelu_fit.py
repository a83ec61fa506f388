"""Coefficients of the GELU used by the bf16 tensor-core GEMM epilogue (epilogue.cuh, gelu_fast2).

GELU(x) = x * Phi(x) with Phi(x) = 1 - q for x >= 0 and q for x < 0, where
q = Phi(-|x|) = erfc(z) / 2, z = |x| / sqrt(2). Write erfc(z) = exp(-z^2) * erfcx(z): erfcx, the
scaled complementary error function, is smooth and slowly varying on z >= 0, so a polynomial
P(z) of degree 8 with P(0) = 1 fits it well where exp(-z^2) does not make it irrelevant. The fit
minimises max_z exp(-z^2) |P(z) - erfcx(z)| on [0, 5] (the absolute error of q) by iteratively
reweighted least squares on Chebyshev nodes (Lawson's method). Beyond z = 5, exp(-z^2) < 1.4e-11.

Run this file to print the coefficients of q = exp(-z^2) * sum_k c_k z^k (the halving folded in).
"""
import numpy as np
from scipy.special import erfc, erfcx

DEGREE = 8
Z_MAX = 5.0


def fit(degree=DEGREE, z_max=Z_MAX, nodes=6000, iters=80):
    t = np.cos(np.pi * (np.arange(nodes) + 0.5) / nodes)
    z = (t + 1.0) / 2.0 * z_max
    A = z[:, None] ** np.arange(1, degree + 1)[None, :]  # c_0 = 1 is fixed
    target = erfcx(z) - 1.0
    wt = np.exp(-z * z)
    w = wt.copy()
    for _ in range(iters):
        c, *_ = np.linalg.lstsq(A * w[:, None], target * w, rcond=None)
        e = np.abs((A @ c - target) * wt)
        w = w * (1.0 + 3.0 * e / e.max())
    return 0.5 * np.concatenate([[1.0], c])  # q = exp(-z^2) * sum c_k z^k


def q_approx(z, coef):
    p = np.zeros_like(z)
    for ck in coef[::-1]:
        p = p * z + ck
    return np.exp(-z * z) * p


def max_error(coef, z_hi=12.0, n=200001):
    """max |q_approx - erfc(z)/2| over [0, z_hi] with z clamped to 7.5 as in the kernel."""
    z = np.linspace(0.0, z_hi, n)
    zc = np.minimum(z, 7.5)
    return float(np.abs(q_approx(zc, coef) - 0.5 * erfc(z)).max())


if __name__ == "__main__":
    c = fit()
    for k, v in enumerate(c):
        print(f"c{k} = {v:.10e}")
    print(f"max |q - erfc(z)/2| = {max_error(c):.3e}")
