"""The FMA-pipe exponential's polynomial: the constants compiled into the kernel are the ones the
committed fit produces, and the fp32 evaluation (range reduction, Horner with fused multiply-adds,
exponent-field add, emulated exactly on the CPU) stays within its relative-error bound."""

import os
import re
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "attention_mugraph_gb300", "csrc")
sys.path.insert(0, CSRC)
import exp2_poly_fit as fit  # noqa: E402


def kernel_coefficients():
    text = open(os.path.join(CSRC, "ptx.cuh")).read()
    found = dict(re.findall(r"constexpr float kExp2C(\d) = (0x[0-9a-fA-F.]+p[-+]\d+)f;", text))
    return np.array([float.fromhex(found[str(i)]) for i in range(len(found))], dtype=np.float32)


def test_kernel_constants_are_the_fit():
    c = fit.fit()
    k = kernel_coefficients()
    assert k.size == fit.DEGREE + 1
    assert np.array_equal(k, c)  # kExp2C0 .. kExp2C5, lowest degree first like the fit


def exp_emulated(s32, coef32):
    """exp_fma's steps in fp32: t = fma(s, log2e, shifter), r = t - shifter, f = fma(s, log2e, -r)
    (each fused multiply-add exact in double, rounded once), polynomial, exponent add."""
    L = np.float64(np.float32(1.4426950408889634))
    s32 = np.maximum(s32, np.float32(-86.0))
    shifter = np.float64(12582912.0)
    t = (s32.astype(np.float64) * L + shifter).astype(np.float32)
    r = (t.astype(np.float64) - shifter).astype(np.float32)
    f = (s32.astype(np.float64) * L - r.astype(np.float64)).astype(np.float32)
    p = fit.horner_fp32(coef32, f)
    return (p.view(np.int32) + (t.view(np.int32) << 23)).astype(np.int32).view(np.float32)


def test_exp_with_folded_scale_error_bound():
    c = fit.fit()
    s = np.linspace(-20.0, 11.1, 2_000_001).astype(np.float32)
    y = exp_emulated(s, c).astype(np.float64)
    ref = np.exp(s.astype(np.float64))
    # The fp32 rounding of log2(e) adds |s| * 2^-25 relative error to the argument.
    assert np.max(np.abs(y / ref - 1.0)) < 6e-7


def test_relative_error_bound():
    c = fit.fit()
    assert fit.max_rel_error(c, -30.0, 12.0) < 3e-7
    # Integers are exact up to the polynomial's value at f = 0.
    x = np.arange(-20, 12, dtype=np.float32)
    y = fit.exp2_emulated(x, c).astype(np.float64)
    assert np.max(np.abs(y / np.exp2(x.astype(np.float64)) - 1)) < 2e-7


def test_underflow_clamp_is_tiny_and_positive():
    c = fit.fit()
    y = fit.exp2_emulated(np.array([-125.0, -200.0, -1e30], dtype=np.float32), c)
    assert (y > 0).all() and (y < 1e-37).all()
