"""Lloyd-Max scalar codebook for the post-rotation coordinate law (fp64 oracle).

What the write-ups say:
* after the random rotation every coordinate of a unit vector follows
  Beta((d-1)/2, (d-1)/2) on [-1, 1], close to N(0, 1/d) for ordinary head
  sizes (A2A TurboQuant explainer, section "Stage 1"; Qiita TurboQuant
  article, section "Rotate, then quantize");
* because that law is known in advance, an MSE-optimal Lloyd-Max quantizer is
  precomputed per head size and bit-width and applied to every coordinate
  independently (Qiita, same section; A2A, "Stage 1" and "How to implement",
  step "precompute the Lloyd-Max codebook").

The law. With alpha = (d-1)/2 the density on [-1, 1] is
    f(t) = (1 - t^2)^(alpha-1) / B(1/2, alpha),
its CDF is F(t) = I_{(1+t)/2}(alpha, alpha) (regularised incomplete beta), and
its first moment over a cell has the closed form
    int_a^b t f(t) dt = ((1-a^2)^alpha - (1-b^2)^alpha) / (2 alpha B(1/2, alpha)).

Lloyd-Max fixed point (2^bits cells, centroids ascending):
    boundary t_j = (c_j + c_{j+1}) / 2       (nearest-neighbour condition)
    centroid c_i = E[T | t_{i-1} < T < t_i]   (centroid condition)
iterated from the law's equal-mass quantile midpoints until no centroid moves
by more than 64 ulp of the largest one (the special functions' own accuracy
is near 1e-15, so that is where the iteration stops improving; for very large
d, where that floor is higher, it stops once the step stalls). Readings: the
stopping rule and the start are not on the pages; the fixed point is unique
because the density is log-concave. The codebook is
kept exactly symmetric (c_i = -c_{2^b-1-i}), so the middle boundary is 0.

Pinned by: the 1-bit closed form, the Gaussian (Max 1960) limit for large d,
the high-resolution distortion bound, Monte Carlo MSE, and an independent
Gaussian Lloyd-Max solved with scipy.stats in the tests.
"""

import functools

import numpy as np
from scipy import special


def _law(d):
    alpha = 0.5 * (d - 1)
    z = special.beta(0.5, alpha)
    return alpha, z


def cdf(t, d):
    alpha, _ = _law(d)
    return special.betainc(alpha, alpha, 0.5 * (1.0 + np.asarray(t, dtype=np.float64)))


def cell_mass(a, b, d):
    return cdf(b, d) - cdf(a, d)


def cell_first_moment(a, b, d):
    alpha, z = _law(d)
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return ((1.0 - a * a) ** alpha - (1.0 - b * b) ** alpha) / (2.0 * alpha * z)


def _symmetrize(c):
    return 0.5 * (c - c[::-1])


@functools.lru_cache(maxsize=None)
def _lloyd_max_cached(d, bits, tol, max_iter):
    if d < 3:
        raise ValueError("d must be at least 3 for the Beta law")
    if not 1 <= bits <= 8:
        raise ValueError("bits must be in 1..8")
    levels = 1 << bits
    alpha, _ = _law(d)
    # start: midpoints (in probability) of equal-mass cells
    p = (np.arange(levels) + 0.5) / levels
    c = 2.0 * special.betaincinv(alpha, alpha, p) - 1.0
    c = _symmetrize(c)
    best, since_best = np.inf, 0
    for it in range(max_iter):
        t = 0.5 * (c[:-1] + c[1:])
        t[levels // 2 - 1] = 0.0
        edges = np.concatenate(([-1.0], t, [1.0]))
        mass = cell_mass(edges[:-1], edges[1:], d)
        new = cell_first_moment(edges[:-1], edges[1:], d) / mass
        new = _symmetrize(new)
        delta = np.max(np.abs(new - c)) / np.max(np.abs(new))
        c = new
        if delta <= tol:
            break
        # at very large d the special functions' rounding sets a floor above
        # tol; stop once the step has not reached a new low for 200 rounds
        if delta < best:
            best, since_best = delta, 0
        else:
            since_best += 1
            if since_best >= 200 and best < 1e-9:
                break
    else:
        raise RuntimeError("Lloyd-Max did not converge")
    t = 0.5 * (c[:-1] + c[1:])
    t[levels // 2 - 1] = 0.0
    return c, t, it + 1


def lloyd_max(d, bits, tol=64 * np.finfo(np.float64).eps, max_iter=200000):
    """Return (centroids [2^bits], boundaries [2^bits - 1]) as float64 arrays."""
    c, t, _ = _lloyd_max_cached(int(d), int(bits), float(tol), int(max_iter))
    return c.copy(), t.copy()


def distortion(d, bits):
    """Per-coordinate MSE D = E[(T - c[idx(T)])^2] = 1/d - sum_i c_i^2 P_i.

    Uses the centroid condition (E[T c] = E[c^2]) and E[T^2] = 1/d.
    """
    c, t = lloyd_max(d, bits)
    edges = np.concatenate(([-1.0], t, [1.0]))
    mass = cell_mass(edges[:-1], edges[1:], d)
    return 1.0 / d - float(np.sum(c * c * mass))


def bucketize(y, boundaries):
    """idx_i = #{j : y_i >= t_j} (a tie goes to the upper cell)."""
    y = np.asarray(y, dtype=np.float64)
    return np.searchsorted(np.asarray(boundaries), y, side="right").astype(np.int64)
