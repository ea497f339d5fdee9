"""Data-independent random orthogonal rotations (fp64 oracle).

What the write-ups say:
* every K/V vector gets a random orthogonal transform built from the QR
  factorisation of a Gaussian matrix, generated once, independent of data
  (A2A TurboQuant explainer, section "Stage 1: random rotation + PolarQuant";
  Qiita TurboQuant article, section "Rotate, then quantize");
* some implementations approximate it with a Walsh-Hadamard transform
  (Qiita TurboQuant article, section "What you hit when you try it").

Readings taken where the pages are silent:
* dense: G is d x d standard normal (rng.normals(seed, d*d), row-major);
  G = QR; Pi = Q diag(sign(diag R)) so that Pi is Haar distributed; a vector
  is rotated as y = Pi x and un-rotated with Pi^T.
* RHT: one sign layer, Pi = H diag(s) / sqrt(d) with H the Sylvester Hadamard
  matrix H_ij = (-1)^popcount(i & j) and s_i = rng.sign_bits(seed, d); only
  for d a power of two.

Pinned by: orthogonality, the Beta((d-1)/2,(d-1)/2) law of a rotated fixed
unit vector over seeds, scipy's Hadamard matrix, and H H^T = d I.
"""

import numpy as np

from . import rng


def dense_rotation(seed, d):
    """Haar-random orthogonal d x d matrix Pi from the QR of a Gaussian matrix."""
    g = rng.normals(seed, d * d).reshape(d, d)
    q, r = np.linalg.qr(g)  # library Householder QR as one step
    s = np.sign(np.diag(r))
    s[s == 0] = 1.0
    return q * s[None, :]


def sylvester_hadamard(d):
    """H_ij = (-1)^popcount(i & j), d a power of two."""
    if d < 1 or d & (d - 1):
        raise ValueError("RHT needs d to be a power of two")
    i = np.arange(d)
    pc = np.zeros((d, d), dtype=np.int64)
    a = i[:, None] & i[None, :]
    while np.any(a):
        pc += a & 1
        a = a >> 1
    return np.where(pc % 2 == 0, 1.0, -1.0)


def rht_signs(seed, d):
    return rng.sign_bits(seed, d)


def rht_rotation(seed, d):
    """Pi = H diag(s) / sqrt(d) as an explicit matrix."""
    h = sylvester_hadamard(d)
    return h * rht_signs(seed, d)[None, :] / np.sqrt(d)


def make_rotation(seed, d, kind):
    """kind: 'dense' or 'rht'. Returns the explicit fp64 matrix Pi (y = Pi x)."""
    if kind == "dense":
        return dense_rotation(seed, d)
    if kind == "rht":
        return rht_rotation(seed, d)
    raise ValueError(kind)


def fwht(x):
    """Unnormalised fast Walsh-Hadamard transform along the last axis (H x)."""
    x = np.array(x, dtype=np.float64, copy=True)
    d = x.shape[-1]
    h = 1
    while h < d:
        x = x.reshape(x.shape[:-1] + (d // (2 * h), 2, h))
        a = x[..., 0, :].copy()
        b = x[..., 1, :].copy()
        x[..., 0, :] = a + b
        x[..., 1, :] = a - b
        x = x.reshape(x.shape[:-3] + (d,))
        h *= 2
    return x


def rotate(pi, x):
    """y = Pi x for each row x of X (rows are vectors)."""
    return np.asarray(x, dtype=np.float64) @ pi.T


def unrotate(pi, y):
    """x = Pi^T y for each row y."""
    return np.asarray(y, dtype=np.float64) @ pi
