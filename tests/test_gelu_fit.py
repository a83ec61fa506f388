"""The GELU of the bf16 tensor-core GEMM epilogue against the exact erf form (CPU only).

The kernel evaluates Phi(-|x|) = erfc(|x|/sqrt 2)/2 as exp(-x^2/2) times a degree-6 polynomial in
min(|x|, 16) whose coefficients gelu_fit.py derives, and GELU(x) = x/2 + |x| (1/2 - q); these
tests re-derive the coefficients, check that the copy in epilogue.cuh is the derived one, bound
the error against scipy's erfc, and replay the kernel's float32 operation order.
"""
import importlib.util
import os
import re

import numpy as np
from scipy.special import erf

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "jepa_vision_encoder_gb300", "csrc")


def load_fit():
    spec = importlib.util.spec_from_file_location("gelu_fit", os.path.join(CSRC, "gelu_fit.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def source_coefficients():
    text = open(os.path.join(CSRC, "epilogue.cuh")).read()
    m = re.search(r"constexpr float c\[7\] = \{([^}]*)\}", text)
    assert m, "coefficient table not found in epilogue.cuh"
    return np.array([float(t.strip().rstrip("f")) for t in m.group(1).split(",")])


def exact_gelu(x):
    return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))


def test_source_coefficients_are_the_fit():
    fit = load_fit()
    c = fit.coefficients_in_x(fit.fit())
    src = source_coefficients()
    assert src.shape == c.shape
    np.testing.assert_allclose(src, c, rtol=2e-9, atol=1e-12)
    assert src[0] == 0.5  # Phi(0) = 1/2 exactly


def test_fit_error_bound():
    fit = load_fit()
    assert fit.max_error(source_coefficients()) <= 1.8e-5


def test_gelu_from_the_source_coefficients_matches_erf_gelu():
    c = source_coefficients().astype(np.float32).astype(np.float64)  # the kernel holds fp32 copies
    fit = load_fit()
    x = np.linspace(-24.0, 24.0, 480001)
    q = fit.q_of_x(x, c)
    g = 0.5 * x + np.abs(x) * (0.5 - q)
    assert np.all(np.abs(g - exact_gelu(x)) <= 1.8e-5 * np.maximum(np.abs(x), 1e-3))
    assert g[np.argmin(np.abs(x))] == 0.0
    assert np.all(g[x >= 16.0] == x[x >= 16.0]) and np.all(g[x <= -16.0] == 0.0)


def test_float32_operation_order_of_the_kernel():
    """The kernel's steps in float32 (exp2 in float64, then rounded): within the bound plus a few ulp."""
    c = source_coefficients().astype(np.float32)
    x = np.linspace(-20.0, 20.0, 200001).astype(np.float32)
    ax = np.abs(x)
    a = np.minimum(ax, np.float32(16.0))
    t = (x * x) * np.float32(-0.72134752044448170)
    p = np.full_like(x, c[6])
    for k in range(5, -1, -1):
        p = (p * a + c[k]).astype(np.float32)
    e = np.exp2(t.astype(np.float64)).astype(np.float32)
    q = p * e
    h = np.float32(0.5) - q
    g = (ax * h + x * np.float32(0.5)).astype(np.float64)
    ref = exact_gelu(x.astype(np.float64))
    # the fit's bound |x| |dq| plus float32 rounding of the few operations (a few ulp of |x| / 2)
    assert np.all(np.abs(g - ref) <= (1.8e-5 + 4e-7) * np.abs(x) + 1e-30)
