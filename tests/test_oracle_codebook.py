"""Pins for the oracle's Lloyd-Max codebook of the Beta law (CPU only)."""

import json
import os

import numpy as np
import pytest
from scipy import integrate, special, stats

from conftest import GOLDEN
from oracle import codebook


@pytest.mark.parametrize("d", [16, 128, 200])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_symmetric_and_sorted(d, bits):
    c, t = codebook.lloyd_max(d, bits)
    assert np.array_equal(c, -c[::-1])
    assert np.all(np.diff(c) > 0) and np.all(np.diff(t) > 0)
    assert t[len(t) // 2] == 0.0
    assert np.all((c[:-1] < t) & (t < c[1:]))


@pytest.mark.parametrize("d", [16, 128, 200])
def test_one_bit_closed_form(d):
    """1 bit: the centroid is E|T| = Gamma(d/2) / (sqrt(pi) Gamma((d+1)/2))."""
    c, _ = codebook.lloyd_max(d, 1)
    want = np.exp(special.gammaln(d / 2) - special.gammaln((d + 1) / 2)) / np.sqrt(np.pi)
    assert abs(c[1] - want) < 1e-13


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_large_d_limit_is_max_gaussian_table(bits):
    """sqrt(d) * codebook -> Max's (1960) Gaussian Lloyd-Max levels as d grows."""
    table = json.load(open(os.path.join(GOLDEN, "max1960_gaussian.json")))
    d = 2**20
    c, _ = codebook.lloyd_max(d, bits)
    got = c[len(c) // 2:] * np.sqrt(d)
    assert np.max(np.abs(got - np.array(table[str(bits)]))) < 2e-4


def _gaussian_lloyd_max(bits, iters=4000):
    """Independent solver: Lloyd-Max for N(0,1) with scipy.stats integrals."""
    levels = 2**bits
    c = stats.norm.ppf((np.arange(levels) + 0.5) / levels)
    for _ in range(iters):
        t = np.concatenate(([-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]))
        mass = stats.norm.cdf(t[1:]) - stats.norm.cdf(t[:-1])
        mom = stats.norm.pdf(t[:-1]) - stats.norm.pdf(t[1:])
        c = mom / mass
    return c


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_large_d_matches_independent_gaussian_solver(bits):
    d = 2**20
    c, _ = codebook.lloyd_max(d, bits)
    g = _gaussian_lloyd_max(bits)
    assert np.max(np.abs(c * np.sqrt(d) - g)) < 1e-4


@pytest.mark.parametrize("d", [128, 200])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_distortion_between_lower_bound_and_high_resolution_bound(d, bits):
    """4^-b <= d * D_b <= (sqrt(3) pi / 2) 4^-b, the "about 2.7x" gap the Qiita page quotes."""
    dd = d * codebook.distortion(d, bits)
    assert 4.0**-bits <= dd <= np.sqrt(3) * np.pi / 2 * 4.0**-bits


@pytest.mark.parametrize("bits", [2, 3])
def test_distortion_by_independent_quadrature_and_optimality(bits):
    """D by scipy quad of (t - c[idx(t)])^2 f(t); perturbed codebooks do worse."""
    d = 128
    c, t = codebook.lloyd_max(d, bits)
    a = (d - 1) / 2
    law = stats.beta(a, a, loc=-1, scale=2)
    edges = np.concatenate(([-1.0], t, [1.0]))

    def dist(cc):
        tot = 0.0
        for i in range(len(cc)):
            v, _ = integrate.quad(lambda x: (x - cc[i]) ** 2 * law.pdf(x), edges[i], edges[i + 1],
                                  epsabs=1e-16, epsrel=1e-12, limit=200)
            tot += v
        return tot

    d0 = dist(c)
    assert abs(d0 - codebook.distortion(d, bits)) < 1e-12
    for i in range(len(c)):
        for eps in (-2e-3, 2e-3):
            cc = c.copy()
            cc[i] += eps / np.sqrt(d)
            assert dist(cc) > d0


def test_monte_carlo_mse_matches_distortion():
    d, bits, n = 128, 3, 2_000_000
    c, t = codebook.lloyd_max(d, bits)
    a = (d - 1) / 2
    y = 2.0 * np.random.default_rng(9).beta(a, a, size=n) - 1.0
    err = (y - c[codebook.bucketize(y, t)]) ** 2
    assert abs(err.mean() - codebook.distortion(d, bits)) < 4 * err.std() / np.sqrt(n)


def test_bucketize_ties_go_up():
    _, t = codebook.lloyd_max(128, 2)
    idx = codebook.bucketize(np.array([t[0], t[1], t[2], -1.0, 1.0]), t)
    assert idx.tolist() == [1, 2, 3, 0, 3]
