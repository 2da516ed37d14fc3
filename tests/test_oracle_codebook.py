"""Pins for the k3v4_nc key codebook (8-level Lloyd-Max for N(0, 1/D)).

Lloyd's optimality conditions are re-checked by numerical quadrature (scipy),
an independent route from the oracle's closed-form cell means; the levels and
the distortion are compared with the textbook table."""
import os

import numpy as np
import pytest
from scipy import integrate, stats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "lloyd_max_gaussian_8level.txt")


def _golden():
    out = {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if "=" in line:
            k, v = line.split("=", 1)
            out[k.strip()] = [float(t) for t in v.split()]
    return out


def _cells(c):
    b = np.concatenate([[-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]])
    return b


def test_converges(oracle_lib):
    c, it = oracle_lib.lloyd_max8()
    assert it > 0
    assert np.all(np.diff(c) > 0)


def test_lloyd_conditions_by_quadrature(oracle_lib):
    c, _ = oracle_lib.lloyd_max8()
    b = _cells(c)
    for m in range(8):
        lo, hi = b[m], b[m + 1]
        num = integrate.quad(lambda x: x * stats.norm.pdf(x), lo, hi, epsabs=1e-14, epsrel=1e-13)[0]
        den = integrate.quad(stats.norm.pdf, lo, hi, epsabs=1e-14, epsrel=1e-13)[0]
        assert abs(num / den - c[m]) < 1e-9


def test_matches_textbook_table(oracle_lib):
    g = _golden()
    c, _ = oracle_lib.lloyd_max8()
    assert np.allclose(c[4:], g["levels"], atol=6e-4)
    assert np.allclose(-c[:4][::-1], g["levels"], atol=6e-4)
    b = _cells(c)[1:-1]
    assert np.allclose(b[3:], g["boundaries"], atol=6e-4)
    mse = 0.0
    bb = _cells(c)
    for m in range(8):
        mse += integrate.quad(lambda x: (x - c[m]) ** 2 * stats.norm.pdf(x), bb[m], bb[m + 1],
                              epsabs=1e-14)[0]
    assert abs(mse - g["mse"][0]) < 5e-5


def test_symmetric(oracle_lib):
    c, _ = oracle_lib.lloyd_max8()
    assert np.allclose(c, -c[::-1], atol=1e-14, rtol=0)
    cb = oracle_lib.codebook16().view(np.float16).astype(np.float64)
    assert np.array_equal(cb, -cb[::-1])


def test_fp16_codebook_is_scaled_levels(oracle_lib):
    c, _ = oracle_lib.lloyd_max8()
    cb = oracle_lib.codebook16()
    ref = (c / np.sqrt(128.0)).astype(np.float16).view(np.uint16)
    assert np.array_equal(cb, ref)
    assert np.all(np.diff(cb.view(np.float16).astype(np.float64)) > 0)


@pytest.mark.parametrize("m", range(7))
def test_boundaries_are_exact_fp32_midpoints(oracle_lib, m):
    cb = oracle_lib.codebook16().view(np.float16).astype(np.float64)
    mid = 0.5 * (cb[m] + cb[m + 1])
    assert float(np.float32(mid)) == mid  # exactly representable: no rounding in the boundary
