"""The GELU of the bf16 tensor-core GEMM epilogue against the exact erf form (CPU only).

The kernel evaluates Phi(-|x|) = erfc(|x|/sqrt 2)/2 as exp(-z^2) times a degree-8 polynomial whose
coefficients gelu_fit.py derives; these tests re-derive them, check that the copy in
epilogue.cuh is the derived one, and bound the error against scipy's erfc.
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
    m = re.search(r"constexpr float c\[9\] = \{([^}]*)\}", text)
    assert m, "coefficient table not found in epilogue.cuh"
    return np.array([float(t.strip().rstrip("f")) for t in m.group(1).split(",")])


def test_source_coefficients_are_the_fit():
    fit = load_fit()
    c = fit.fit()
    src = source_coefficients()
    assert src.shape == c.shape
    np.testing.assert_allclose(src, c, rtol=2e-9, atol=1e-12)
    assert src[0] == 0.5  # Phi(0) = 1/2 exactly


def test_fit_error_bound():
    fit = load_fit()
    assert fit.max_error(source_coefficients()) <= 1.2e-6


def test_gelu_from_the_source_coefficients_matches_erf_gelu():
    c = source_coefficients().astype(np.float32).astype(np.float64)  # the kernel holds fp32 copies
    fit = load_fit()
    x = np.linspace(-12.0, 12.0, 240001)
    z = np.minimum(np.abs(x) / np.sqrt(2.0), 7.5)
    q = fit.q_approx(z, c)
    g = x * np.where(x >= 0.0, 1.0 - q, q)
    exact = 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))
    assert np.all(np.abs(g - exact) <= 1.3e-6 * np.maximum(np.abs(x), 1e-3))
    assert g[np.argmin(np.abs(x))] == 0.0
