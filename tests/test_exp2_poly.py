"""The polynomial exponential of the prefill softmax, checked on the CPU: its coefficients
are the fit that exp2_poly_fit.py derives, the fit meets its relative-error bound against
numpy's exp2, and the range reduction (rint by adding 1.5 * 2^23, then r added to the
exponent field) reproduces 2^x over the range the softmax feeds it."""
import os
import re
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "tiled_attention_06_gb300", "csrc")
sys.path.insert(0, CSRC)

import exp2_poly_fit  # noqa: E402


def header_coeffs():
    with open(os.path.join(CSRC, "fa_ptx.cuh")) as f:
        src = f.read()
    body = src[src.index("exp2_poly_x2"):]
    return np.array([float(re.search(rf"kC{k} = ([-+0-9.e]+)f", body).group(1)) for k in range(4)],
                    dtype=np.float32)


def fma32(a, b, c):
    # products of two float32 values are exact in float64; one rounding to float32
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def poly_exp2_f32(x):
    """The device routine's steps in float32 arithmetic."""
    c = header_coeffs()
    shift = np.float32(12582912.0)
    x = np.maximum(x.astype(np.float32), np.float32(-126.0))
    t = (x + shift).astype(np.float32)
    r = (t - shift).astype(np.float32)
    f = fma32(r, np.full_like(r, -1.0), x)
    p = fma32(np.full_like(f, c[3]), f, np.full_like(f, c[2]))
    p = fma32(p, f, np.full_like(f, c[1]))
    p = fma32(p, f, np.full_like(f, c[0]))
    bits = p.view(np.uint32) + (t.view(np.uint32) << np.uint32(23))
    return bits.view(np.float32), f, r


def test_header_coefficients_are_the_fit():
    c, err = exp2_poly_fit.fit(3)
    assert np.allclose(header_coeffs(), c, rtol=2e-6, atol=0)
    assert err < 7.6e-5


def test_fit_relative_error_bound():
    assert exp2_poly_fit.rel_error(header_coeffs()) < 7.6e-5
    # a degree-3 polynomial cannot do much better: Taylor's fourth term alone, at f = 1/2,
    # is (ln 2 / 2)^4 / 24 = 6e-4, so the minimax fit must sit between 1e-5 and that
    assert exp2_poly_fit.rel_error(header_coeffs()) > 1e-5


def test_range_reduction_is_exact():
    x = np.linspace(-126.0, 9.0, 270001).astype(np.float32)
    _, f, r = poly_exp2_f32(x)
    assert np.array_equal(r, np.rint(x))  # rint: ties to even, as the float32 add rounds
    assert np.all(np.abs(f) <= 0.5)
    assert np.array_equal(f.astype(np.float64), x.astype(np.float64) - np.rint(x))


@pytest.mark.parametrize("lo,hi", [(-125.0, 9.0), (-20.0, 0.0), (-1.0, 1.0)])
def test_matches_exp2(lo, hi):
    x = np.linspace(lo, hi, 400003).astype(np.float32)
    y, _, _ = poly_exp2_f32(x)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y.astype(np.float64) / ref - 1.0)
    assert rel.max() < 8e-5  # fit bound plus float32 rounding of the polynomial


def test_clamp_keeps_tiny_results_tiny_and_nonnegative():
    x = np.array([-126.0, -130.0, -1000.0, -3.0e6], dtype=np.float32)
    y, _, _ = poly_exp2_f32(x)
    assert np.all(y >= 0) and np.all(y < 2.0 ** -125)
