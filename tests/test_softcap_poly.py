"""The softcap polynomials in csrc/common.cuh against numpy's tanh.

tanh(y) = y * (1 + t * R(t)), t = y^2, serves |y| <= kTanhPolyY in the
kernels; larger |y| fall back to the exp-based tanh.  The forward also has a
linear R for |y| <= kTanhShortY.  Their error must stay at fp32 rounding level
there, and R's leading coefficient must be positive (a score of -inf then stays
-inf through the polynomial form)."""
import os
import re

import numpy as np

CSRC = os.path.join(os.path.dirname(__file__), "..", "attention_attn_fwd_08_gb300", "csrc")
SRC = os.path.join(CSRC, "common.cuh")


def _consts():
    s = open(SRC).read()
    y0 = float(re.search(r"kTanhPolyY\s*=\s*([-0-9.eE+]+)f", s).group(1))
    r = [float(re.search(r"kTanhR%d\s*=\s*([-0-9.eE+]+)f" % i, s).group(1)) for i in range(4)]
    return y0, r


def _poly_f32(y, r):
    y = y.astype(np.float32)
    t = y * y
    p = np.float32(r[3])
    for c in (r[2], r[1], r[0]):
        p = p * t + np.float32(c)
    return y + y * (t * p)


def test_poly_matches_tanh_in_range():
    y0, r = _consts()
    y = np.linspace(-y0, y0, 400001)
    ref = np.tanh(y.astype(np.float32).astype(np.float64))
    got = _poly_f32(y, r).astype(np.float64)
    nz = np.abs(ref) > 1e-30
    rel = np.max(np.abs(got[nz] - ref[nz]) / np.abs(ref[nz]))
    assert rel < 3e-7, rel  # a few fp32 ulp
    # the fit itself (exact arithmetic) is below 2e-8
    yy = np.linspace(1e-6, y0, 100001)
    t = yy * yy
    fit = yy * (1 + t * np.polyval(r[::-1], t))
    assert np.max(np.abs(fit / np.tanh(yy) - 1)) < 2e-8


def test_poly_is_odd_and_leading_coefficient_positive():
    y0, r = _consts()
    y = np.linspace(0, y0, 1001)
    assert np.array_equal(_poly_f32(-y, r), -_poly_f32(y, r))
    assert r[3] > 0 and r[0] < 0  # R(0) = -1/3 to first order
    assert abs(r[0] + 1 / 3) < 1e-5


def _short_consts():
    s = open(SRC).read()
    y0 = float(re.search(r"kTanhShortY\s*=\s*([-0-9.eE+]+)f", s).group(1))
    r = [float(re.search(r"kTanhS%d\s*=\s*([-0-9.eE+]+)f" % i, s).group(1)) for i in range(2)]
    return y0, r


def test_short_poly_matches_tanh_in_range():
    y0, r = _short_consts()
    assert y0 < _consts()[0]  # serves a sub-range of the cubic's
    y = np.linspace(-y0, y0, 400001).astype(np.float32)
    t = y * y
    got = (y + y * (t * (np.float32(r[1]) * t + np.float32(r[0])))).astype(np.float64)
    ref = np.tanh(y.astype(np.float64))
    nz = np.abs(ref) > 1e-30
    assert np.max(np.abs(got[nz] - ref[nz]) / np.abs(ref[nz])) < 3e-7
    yy = np.linspace(1e-6, y0, 100001)
    tt = yy * yy
    assert np.max(np.abs(yy * (1 + tt * (r[0] + r[1] * tt)) / np.tanh(yy) - 1)) < 1e-8
    assert r[1] > 0 and abs(r[0] + 1 / 3) < 1e-5 and abs(r[1] - 2 / 15) < 5e-3  # tanh's Taylor terms
