"""The numeric constants typed into the gated-unit kernels are the published ones.

The bf16 GeLU-erf path takes the normal CDF from the rational approximation of
erfc in Abramowitz & Stegun, Handbook of Mathematical Functions, formula 7.1.26,
whose error bound (|erf error| < 1.5e-7) is far inside the bf16 parity bound.
A slip in one of its coefficients could stay inside the bf16 bound too, so the
GPU parity tests would not see it.  This test reads the constants from the
kernel source and checks them against their definitions, and the formula built
from them against scipy's erf: in float64 within the published bound, and
evaluated in float32 (as the kernel does) within a small multiple of it.  CPU only.
"""

import math
import os
import re

import numpy as np
from scipy.special import erf

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "rmsnorm_fwd_bwd_03_gb300", "csrc", "glu.cu")


def _constants():
    with open(SRC, encoding="utf-8") as f:
        text = f.read()
    out = {}
    for name, val in re.findall(r"\b(k[A-Z][A-Za-z0-9]*)\s*=\s*(-?[0-9.]+(?:e-?[0-9]+)?)f\b", text):
        out[name] = float(val)
    return out


def test_gelu_constants_match_their_definitions():
    c = _constants()
    f32 = lambda v: float(np.float32(v))  # noqa: E731
    assert f32(c["kGeluK"]) == f32(2.0 * math.sqrt(2.0 / math.pi))
    assert c["kGeluC"] == 0.044715
    assert f32(c["kInvSqrt2"]) == f32(1.0 / math.sqrt(2.0))
    assert f32(c["kInvSqrt2Pi"]) == f32(1.0 / math.sqrt(2.0 * math.pi))
    # e^a = 2^(a log2 e) in the bf16 exponentials
    assert f32(c["kLog2e"]) == f32(1.0 / math.log(2.0))


def _as_erfc(z, c, dtype):
    z = np.asarray(z, dtype=dtype)
    one = dtype(1.0)
    t = one / (one + dtype(c["kAsP"]) * z)
    poly = t * (dtype(c["kAsA1"]) + t * (dtype(c["kAsA2"]) + t * (dtype(c["kAsA3"]) + t * (
        dtype(c["kAsA4"]) + t * dtype(c["kAsA5"])))))
    return poly * np.exp(-z * z)


def test_abramowitz_stegun_coefficients_meet_the_published_bound():
    c = _constants()
    z = np.linspace(0.0, 10.0, 200001)
    err = np.max(np.abs((1.0 - _as_erfc(z, c, np.float64)) - erf(z)))
    assert err < 1.5e-7, err


def test_gelu_erf_in_float32_from_these_constants():
    # x * Phi(x) with Phi from the formula, all in float32 as in the kernel
    # (the kernel's fast exponential and division add a few float32 ulps; the
    # bound below is for float32 library exp and division).
    c = _constants()
    x = np.linspace(-12.0, 12.0, 480001).astype(np.float32)
    z = np.abs(x) * np.float32(c["kInvSqrt2"])
    half_erfc = np.float32(0.5) * _as_erfc(z, c, np.float32)
    cdf = np.where(x >= 0, np.float32(1.0) - half_erfc, half_erfc)
    gelu = (x * cdf).astype(np.float64)
    x64 = x.astype(np.float64)
    exact = 0.5 * x64 * (1.0 + erf(x64 / math.sqrt(2.0)))
    err = np.max(np.abs(gelu - exact))
    assert err < 1e-6, err
