"""Pins for the oracle's random streams and rotations (CPU only)."""

import os

import numpy as np
import pytest
import scipy.linalg
import scipy.stats
import torch

from conftest import GOLDEN
from oracle import rng, rotation


def test_splitmix64_known_answer():
    want = [int(line, 16) for line in open(os.path.join(GOLDEN, "splitmix64_seed0.txt"))
            if line.strip() and not line.startswith("#")]
    got = [int(v) for v in rng.splitmix64(0, len(want))]
    assert got == want


def test_splitmix64_counter_form_matches_sequential_offsets():
    # draw k of a stream must not depend on how many draws were requested
    a = rng.splitmix64(12345, 100)
    b = rng.splitmix64(12345, 50, start=50)
    assert np.array_equal(a[50:], b)


def test_normals_distribution():
    z = rng.normals(7, 400_000)
    assert abs(z.mean()) < 4 / np.sqrt(z.size)
    assert abs(z.var() - 1) < 4 * np.sqrt(2 / z.size)
    assert scipy.stats.kstest(z, "norm").pvalue > 1e-3


def test_uniforms_range_and_sign_balance():
    u = rng.uniforms(3, 100_000)
    assert u.min() >= 0 and u.max() < 1
    assert scipy.stats.kstest(u, "uniform").pvalue > 1e-3
    s = rng.sign_bits(3, 100_000)
    assert set(np.unique(s)) == {-1.0, 1.0}
    assert abs(s.mean()) < 4 / np.sqrt(s.size)


def test_bf16_rounding_matches_torch():
    x = rng.normals(11, 20000).astype(np.float32).astype(np.float64)
    # add exact ties: values halfway between bf16 neighbours
    ties = np.array([1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8, -2.0 - 2.0**-7, 3.0 + 2.0**-7])
    x = np.concatenate([x, ties])
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(rng.round_to_bf16(x), want)


@pytest.mark.parametrize("d", [16, 128, 200])
def test_dense_rotation_orthogonal(d):
    pi = rotation.dense_rotation(1, d)
    assert np.max(np.abs(pi.T @ pi - np.eye(d))) < 1e-12
    assert np.max(np.abs(pi @ pi.T - np.eye(d))) < 1e-12


def test_dense_rotation_is_haar_on_a_fixed_vector():
    """A rotated fixed unit vector has Beta((d-1)/2,(d-1)/2) coordinates on [-1,1].

    Over many seeds y_0 = (Pi e_0)_0 must follow the law (a QR without the
    sign fix gives y_0 < 0 always and fails here); moments E y^2 = 1/d,
    E y^4 = 3/(d(d+2)).
    """
    d, seeds = 12, 4000
    x = np.zeros(d)
    x[0] = 1.0
    y0 = np.array([rotation.dense_rotation(s, d) @ x for s in range(seeds)])[:, 0]
    a = (d - 1) / 2
    law = scipy.stats.beta(a, a, loc=-1, scale=2)
    assert scipy.stats.kstest(y0, law.cdf).pvalue > 1e-3
    m2, m4 = np.mean(y0**2), np.mean(y0**4)
    se2 = np.std(y0**2) / np.sqrt(seeds)
    se4 = np.std(y0**4) / np.sqrt(seeds)
    assert abs(m2 - 1 / d) < 4 * se2
    assert abs(m4 - 3 / (d * (d + 2))) < 4 * se4


def test_rotation_spreads_outliers():
    """Energy of outlier channels is spread over all coordinates after rotation."""
    d = 128
    x = np.ones(d)
    x[[3, 40, 77, 100]] = 20.0
    x /= np.linalg.norm(x)
    assert np.max(np.abs(x)) > 0.45
    for kind in ("dense", "rht"):
        y = rotation.make_rotation(1, d, kind) @ x
        assert np.max(np.abs(y)) < 5.0 / np.sqrt(d)


def test_sylvester_matches_scipy_hadamard():
    for d in (2, 8, 64, 128, 256):
        assert np.array_equal(rotation.sylvester_hadamard(d), scipy.linalg.hadamard(d))


def test_hadamard_orthogonality_and_fwht():
    d = 128
    h = rotation.sylvester_hadamard(d)
    assert np.array_equal(h @ h.T, d * np.eye(d))
    x = rng.normals(5, 3 * d).reshape(3, d)
    assert np.max(np.abs(rotation.fwht(x) - x @ h.T)) < 1e-12
    pi = rotation.rht_rotation(1, d)
    assert np.max(np.abs(pi @ pi.T - np.eye(d))) < 1e-12
    s = rotation.rht_signs(1, d)
    assert np.max(np.abs(rotation.rotate(pi, x) - rotation.fwht(x * s) / np.sqrt(d))) < 1e-12


def test_rht_rejects_non_power_of_two():
    with pytest.raises(ValueError):
        rotation.rht_rotation(1, 200)
