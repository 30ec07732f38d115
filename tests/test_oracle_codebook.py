"""Pins for the oracle's Lloyd-Max codebook ("centroids.py" section of the
vLLM PR 38479 digest).  None of these re-types the oracle's formula: they
check it against closed forms of the Gaussian integrals (erf), the known
1-bit optimum, symmetry, and a Lloyd iteration written with scipy's
normal CDF instead of trapezoid sums."""
import math

import numpy as np
import pytest
from scipy.special import erf
from scipy.stats import norm as gauss


def _closed_form_means(edges, sigma):
    """E[X | a < X < b] for X ~ N(0, sigma^2), exactly."""
    a, b = np.asarray(edges[:-1]), np.asarray(edges[1:])
    pdf = lambda x: np.exp(-x * x / (2 * sigma**2)) / math.sqrt(2 * math.pi * sigma**2)
    cdf = lambda x: 0.5 * (1 + erf(x / (sigma * math.sqrt(2))))
    return sigma**2 * (pdf(a) - pdf(b)) / (cdf(b) - cdf(a))


def _scipy_lloyd(bits, sigma, iters=20000):
    """Plain Lloyd iteration with exact conditional means on the real line."""
    n = 1 << bits
    c = np.linspace(-3.5 * sigma, 3.5 * sigma, n + 1)
    c = 0.5 * (c[:-1] + c[1:])
    for _ in range(iters):
        e = np.concatenate([[-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]])
        a, b = e[:-1], e[1:]
        num = sigma**2 * (gauss.pdf(a, scale=sigma) - gauss.pdf(b, scale=sigma))
        den = gauss.cdf(b, scale=sigma) - gauss.cdf(a, scale=sigma)
        nc = num / den
        if np.max(np.abs(nc - c)) < 1e-15:
            c = nc
            break
        c = nc
    return c


@pytest.mark.parametrize("d", [64, 128, 256])
def test_one_bit_is_sqrt_2_over_pi(orc, d):
    sigma = 1 / math.sqrt(d)
    _, c32, m32, _ = orc.lloyd_max(d, 1)
    target = math.sqrt(2 / math.pi) * sigma
    # page's 200-panel trapezoid on [0, 10.5 sigma]: within 5e-4 relative
    assert abs(c32[1] - target) / target < 5e-4
    assert abs(c32[0] + target) / target < 5e-4
    # the same algorithm with 100x the panels: the trapezoid error falls as
    # h^2, so 1e4 times smaller
    c64, _, _, _ = orc.lloyd_max(d, 1, trapz_n=20000, max_iter=5000)
    assert abs(c64[1] - target) / target < 5e-8


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_fixed_point_conditional_means(orc, bits):
    d = 128
    sigma = 1 / math.sqrt(d)
    c64, _, _, it = orc.lloyd_max(d, bits)
    edges = np.concatenate([[-10.5 * sigma], 0.5 * (c64[:-1] + c64[1:]), [10.5 * sigma]])
    exact = _closed_form_means(edges, sigma)
    # 200 panels + at most 200 iterations: residual within 2e-3 relative
    assert np.max(np.abs(exact - c64) / np.abs(exact)) < 2e-3
    # fine panels and enough iterations: the fixed point of the exact map
    c64f, _, _, _ = orc.lloyd_max(d, bits, trapz_n=20000, max_iter=20000, tol=1e-14)
    ref = _scipy_lloyd(bits, sigma)
    # (trapezoid error at 20000 panels is ~1e-8 relative, as in the 1-bit case)
    assert np.max(np.abs(c64f - ref)) / sigma < 5e-7


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_symmetry_and_order(orc, bits):
    _, c32, m32, _ = orc.lloyd_max(128, bits)
    assert np.all(np.diff(c32) > 0)
    assert np.max(np.abs(c32 + c32[::-1])) < 1e-7
    # midpoints: fp32 mean of fp32 neighbours, strictly between them
    assert np.all(m32 > c32[:-1]) and np.all(m32 < c32[1:])
    exact_mid = (c32[:-1].astype(np.float64) + c32[1:].astype(np.float64)) / 2
    assert np.array_equal(m32, exact_mid.astype(np.float32))


def test_matches_gaussian_quantizer_tables(orc):
    """Unit-variance optimum re-derived with exact integrals (the Gaussian
    Lloyd-Max quantizer of Max, 1960): the page's algorithm lands within
    2e-3 of it in units of sigma at 2-4 bits."""
    for bits in (2, 3, 4):
        ref = _scipy_lloyd(bits, 1.0)
        _, c32, _, _ = orc.lloyd_max(128, bits)
        assert np.max(np.abs(c32 * math.sqrt(128) - ref)) < 2e-3, bits


def test_iteration_cap_and_previous_iterate(orc):
    """The loop stops at 200 iterations; at an earlier stop the kept iterate
    is the one before the last update (its move is below tol)."""
    _, _, _, it4 = orc.lloyd_max(128, 4)
    assert it4 == 200
    c_a, _, _, it1 = orc.lloyd_max(128, 1)
    assert it1 < 200
    c_b, _, _, _ = orc.lloyd_max(128, 1, max_iter=it1 + 1)
    assert np.array_equal(c_a, c_b)


def test_page_constants(orc):
    """The oracle runs with the constants the page's centroids.py prints:
    its defaults are the golden file's panel count, iteration cap and
    tolerance, and with no iteration it returns the page's start, the
    centres of 2^b equal cells on [-3.5 sigma, 3.5 sigma]."""
    import inspect
    vals = {}
    with open(__file__.replace("test_oracle_codebook.py", "golden/page_numbers.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    defaults = inspect.signature(orc.lloyd_max).parameters
    assert defaults["trapz_n"].default == vals["lloyd_trapz_panels"]
    assert defaults["max_iter"].default == vals["lloyd_max_iter"]
    assert defaults["tol"].default == vals["lloyd_tol"]
    for d, bits in ((128, 3), (64, 2)):
        sigma = 1 / math.sqrt(d)
        half = vals["lloyd_init_range_sigmas"] * sigma
        n = 1 << bits
        c0, _, _, it = orc.lloyd_max(d, bits, max_iter=0)
        assert it == 0
        start = -half + 2 * half * (np.arange(n) + 0.5) / n
        assert np.max(np.abs(c0 - start)) < 1e-15
