"""The soft split's normal distribution function in the compositing kernels
(Abramowitz and Stegun, Handbook of Mathematical Functions, 26.2.17) against
scipy's ndtr: the constants are read from the kernel source, and the formula
evaluated with them must stay within the handbook's bound (|error| < 7.5e-8)
everywhere, in double; in single precision, as the kernels evaluate it, within
a few 1e-7.  A mistyped constant or a wrong sign fails the first check."""

import os
import re

import numpy as np
from scipy.special import ndtr

SRC = os.path.join(os.path.dirname(__file__), "..", "differentiable_hybrid_mesh_tile_b300", "csrc",
                   "gm_composite.cu")


def _constants():
    text = open(SRC).read()
    body = text[text.index("normal_cdf(float x)"):]
    body = body[:body.index("}")]
    vals = dict((k, float(v)) for k, v in re.findall(r"\b(P|B[1-5])\s*=\s*(-?[0-9.]+)f", body))
    assert sorted(vals) == ["B1", "B2", "B3", "B4", "B5", "P"], vals
    return vals


def _phi(x, k, dtype):
    x = np.asarray(x, dtype)
    one = dtype(1.0)
    ax = np.abs(x)
    t = one / (dtype(k["P"]) * ax + one)
    poly = t * (dtype(k["B1"]) + t * (dtype(k["B2"]) + t * (dtype(k["B3"]) + t * (dtype(k["B4"]) +
                                                                                 t * dtype(k["B5"])))))
    q = dtype(0.3989422804014327) * np.exp(dtype(-0.5) * ax * ax) * poly
    return np.where(x >= 0, one - q, q)


def test_normal_cdf_within_the_handbook_bound():
    k = _constants()
    x = np.linspace(-9.0, 9.0, 720001)
    err = np.abs(_phi(x, k, np.float64) - ndtr(x))
    assert err.max() < 7.5e-8, err.max()
    # down to the split's tail (f(-3) = 0.00135; below -2.75 the kernels skip the pair)
    # the relative error stays small: the tail is formed directly, without cancellation
    xt = np.linspace(-3.0, 0.0, 3001)
    rel = np.abs(_phi(xt, k, np.float64) / ndtr(xt) - 1.0)
    assert rel.max() < 6e-5, rel.max()


def test_normal_cdf_single_precision():
    k = _constants()
    x = np.linspace(-6.0, 6.0, 120001).astype(np.float32)
    err = np.abs(_phi(x, k, np.float32).astype(np.float64) - ndtr(x.astype(np.float64)))
    assert err.max() < 4e-7, err.max()
