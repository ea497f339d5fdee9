"""PolarQuant key quantization, fp64 oracle (the comparison variant).

What the write-ups say:
* the key vector is taken from Cartesian to polar coordinates, as (x, y) ->
  (r, theta) in two dimensions, applied again and again to pairs of adjacent
  dimensions of the high-dimensional vector (DeepSignal TurboQuant article,
  section "PolarQuant"); the vector is normalised and the dimensions are
  paired recursively, the radius carrying the magnitude and the angles the
  direction (A2A TurboQuant explainer, "Stage 1", PolarQuant bullets);
* the angles are quantized at high precision and the radius at low
  precision; the inverse map is plain trigonometry (DeepSignal, same section);
* the angles' distribution is concentrated and known in advance, so no
  per-block normalisation constants are needed, and a Lloyd-Max quantizer of
  a Beta law maps each value to a few bits (A2A, same bullets);
* it follows the data-independent random rotation (A2A, "Stage 1").

Readings (the pages give no formulas):
* rotation first, as for the other modes: y = Pi x / ||x|| with ||x|| stored as
  float16 (the "radius": the final radius of the recursion is ||y|| = 1, so the
  only radius kept is the vector norm, stored like the other modes' norms);
* d a power of two; level 1 pairs coordinates (y_2i, y_2i+1) into
  rho_1,i = hypot and psi_1,i = atan2(y_2i+1, y_2i) in (-pi, pi]; level l >= 2
  pairs the radii of level l - 1 the same way, psi_l,i in [0, pi/2]; log2(d)
  levels, d - 1 angles in all;
* the angle laws after a Haar rotation: level 1 uniform on the circle; at
  level l >= 2 the two radii are norms of independent k = 2^(l-1) dimensional
  Gaussian blocks (the direction of a Gaussian vector is uniform on the
  sphere), so psi has density proportional to (sin psi cos psi)^(k - 1) on
  [0, pi/2], i.e. sin^2 psi ~ Beta(k/2, k/2) (the page's "Beta law");
* one Lloyd-Max codebook per level for its law (level 1: the uniform law,
  whose optimum has equal cells; the grid starts at -pi); level-1 angles at
  `bits1` bits, higher levels at `bits2` (the default 4 / 2 is 382 bits per
  128-vector, about 3 bits per coordinate, the "3 bits in the main stage" the
  A2A page gives as an example); ties go to the upper cell;
* reconstruction by the inverse recursion from the centroid angles (unit norm
  exactly), keys scored as n <q', y_hat> with q' = Pi q (no sign sketch: the
  plain PolarQuant estimator), values kept in the MSE mode.

Packed layout (this project's specification): the angle codes as one LSB-first
bit stream, level 1 first (angle i at bits1 * i), then levels 2, 3, ... in
order, each angle at its level's width; row stride rounded up to 16 bytes.

Decode (this library's reading, the same as the TurboQuant decode): the key
logits above, p = softmax(scale * l) over the visible tokens (scale 1/sqrt(d)
unless given), a = sum_t p_t nV_t cV[idxV_t] with MSE values, o = Pi^T a.

Pinned by: the exact inverse without quantization; the angle laws against the
empirical angles of Haar-random unit vectors (KS tests); the Lloyd-Max
conditions of every level's codebook, checked with an independent quadrature;
the closed-form distortion of d = 2 (one uniform angle); logits equal to the
dense reconstruction's dot products; a hand-worked packing example; decode
equal to textbook softmax attention over the explicit reconstructions.
"""

import functools

import numpy as np
from scipy import special

from . import attention
from . import quantize as qmod
from . import rotation


def levels(d):
    L = int(round(np.log2(d)))
    if d < 2 or (1 << L) != d:
        raise ValueError("PolarQuant needs d a power of two, d >= 2")
    return L


def angle_count(d):
    """Angles per level: d/2, d/4, ..., 1."""
    return [d >> l for l in range(1, levels(d) + 1)]


def polar(y):
    """Recursive polar transform of rows of y: (list of angle arrays per level, final radius)."""
    y = np.atleast_2d(np.asarray(y, dtype=np.float64))
    rho = y
    angles = []
    for l in range(levels(y.shape[1])):
        a, b = rho[:, 0::2], rho[:, 1::2]
        angles.append(np.arctan2(b, a))
        rho = np.hypot(a, b)
    return angles, rho[:, 0]


def unpolar(angles, radius=None):
    """Inverse recursion: from the top radius (1 if None) down through the angles."""
    n = angles[0].shape[0]
    rho = np.ones((n, 1)) if radius is None else np.asarray(radius, dtype=np.float64).reshape(n, 1)
    for psi in reversed(angles):
        out = np.empty((n, 2 * rho.shape[1]))
        out[:, 0::2] = rho * np.cos(psi)
        out[:, 1::2] = rho * np.sin(psi)
        rho = out
    return rho


# ---------------------------------------------------------------- the laws --
def angle_cdf(psi, level):
    """CDF of the level's angle after a Haar rotation."""
    psi = np.asarray(psi, dtype=np.float64)
    if level == 1:
        return np.clip((psi + np.pi) / (2 * np.pi), 0.0, 1.0)
    k = 1 << (level - 1)
    s = np.clip(np.sin(np.clip(psi, 0.0, np.pi / 2)) ** 2, 0.0, 1.0)
    return special.betainc(0.5 * k, 0.5 * k, s)


def angle_pdf(psi, level):
    psi = np.asarray(psi, dtype=np.float64)
    if level == 1:
        return np.where((psi >= -np.pi) & (psi <= np.pi), 1.0 / (2 * np.pi), 0.0)
    k = 1 << (level - 1)
    # sin^2 psi ~ Beta(k/2, k/2): f(psi) = 2 (sin psi cos psi)^(k-1) / B(k/2, k/2)
    return np.where((psi >= 0) & (psi <= np.pi / 2),
                    2.0 * (np.sin(psi) * np.cos(psi)) ** (k - 1) / special.beta(0.5 * k, 0.5 * k), 0.0)


def angle_range(level):
    return (-np.pi, np.pi) if level == 1 else (0.0, np.pi / 2)


# ------------------------------------------------------------ the codebooks --
@functools.lru_cache(maxsize=None)
def _codebook_cached(level, bits):
    lo, hi = angle_range(level)
    n = 1 << bits
    if level == 1:
        # the uniform law: equal cells (Lloyd-Max optimum), grid from -pi
        w = (hi - lo) / n
        t = lo + w * np.arange(1, n)
        c = lo + w * (np.arange(n) + 0.5)
        return c, t
    # start at equal-mass cell midpoints, then the Lloyd-Max fixed point with
    # the cell mass from the CDF and the first moment by quadrature
    k = 1 << (level - 1)
    p = (np.arange(n) + 0.5) / n
    c = np.arcsin(np.sqrt(special.betaincinv(0.5 * k, 0.5 * k, p)))
    # first moments by 96-point Gauss-Legendre on each cell (the density is
    # smooth and at most a 63rd power of sin cos on a cell of width < pi/2)
    xg, wg = special.roots_legendre(96)
    for _ in range(20000):
        t = 0.5 * (c[:-1] + c[1:])
        edges = np.concatenate(([lo], t, [hi]))
        a, b = edges[:-1, None], edges[1:, None]
        u = 0.5 * (b - a) * xg[None, :] + 0.5 * (a + b)
        mom = 0.5 * (b[:, 0] - a[:, 0]) * np.sum(wg[None, :] * u * angle_pdf(u, level), axis=1)
        mass = angle_cdf(edges[1:], level) - angle_cdf(edges[:-1], level)
        new = mom / mass
        # the law is symmetric about pi/4
        new = 0.5 * (new + (np.pi / 2 - new[::-1]))
        delta = np.max(np.abs(new - c))
        c = new
        if delta < 1e-14:
            break
    else:
        raise RuntimeError("angle Lloyd-Max did not converge")
    t = 0.5 * (c[:-1] + c[1:])
    return c, t


def codebook(level, bits):
    """(centroids [2^bits], boundaries [2^bits - 1]) of the level's angle law."""
    c, t = _codebook_cached(int(level), int(bits))
    return c.copy(), t.copy()


def level_bits(d, bits1, bits2):
    return [bits1] + [bits2] * (levels(d) - 1)


def row_bits(d, bits1, bits2):
    return sum(nb * w for nb, w in zip(angle_count(d), level_bits(d, bits1, bits2)))


# -------------------------------------------------------------- quantize ----
def quantize(x, pi, bits1=4, bits2=2):
    """PolarQuant keys: norm, rotate, polar transform, one codebook per level.

    Returns n (exact norm), norm16, y (rotated unit vectors), angles (fp64, per
    level), idx (codes per level), y_hat (reconstruction, unit norm)."""
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    d = x.shape[1]
    n = np.sqrt(np.sum(x * x, axis=1))
    safe = np.where(n > 0, n, 1.0)
    y = rotation.rotate(pi, x) / safe[:, None]
    y[n == 0] = 0.0
    angles, _ = polar(y)
    idx, cent = [], []
    for l, w in enumerate(level_bits(d, bits1, bits2), start=1):
        c, t = codebook(l, w)
        k = np.searchsorted(t, angles[l - 1], side="right").astype(np.int64)
        idx.append(k)
        cent.append(c[k])
    y_hat = unpolar(cent)
    return {"n": n, "norm16": qmod.fp16_rne(n), "y": y, "angles": angles, "idx": idx, "y_hat": y_hat,
            "bits": (bits1, bits2)}


def pack(idx, d, bits1, bits2):
    """LSB-first stream: level 1 angles, then level 2, ...; stride rounded up to 16 bytes."""
    n = idx[0].shape[0]
    widths = np.concatenate([np.full(cnt, w) for cnt, w in zip(angle_count(d), level_bits(d, bits1, bits2))])
    codes = np.concatenate(idx, axis=1)
    nbits = int(widths.sum())
    stride = qmod.row_stride(nbits)
    out = np.zeros((n, stride), dtype=np.uint8)
    off = np.concatenate(([0], np.cumsum(widths)[:-1]))
    for j in range(codes.shape[1]):
        for b in range(int(widths[j])):
            bit = (codes[:, j] >> b) & 1
            p = off[j] + b
            out[:, p // 8] |= (bit << (p % 8)).astype(np.uint8)
    return out


def unpack(packed, d, bits1, bits2):
    packed = np.atleast_2d(np.asarray(packed, dtype=np.uint8))
    counts, ws = angle_count(d), level_bits(d, bits1, bits2)
    widths = np.concatenate([np.full(cnt, w) for cnt, w in zip(counts, ws)])
    off = np.concatenate(([0], np.cumsum(widths)[:-1]))
    flat = np.zeros((packed.shape[0], widths.size), dtype=np.int64)
    for j in range(widths.size):
        for b in range(int(widths[j])):
            p = off[j] + b
            flat[:, j] |= ((packed[:, p // 8] >> (p % 8)) & 1).astype(np.int64) << b
    out, s = [], 0
    for cnt in counts:
        out.append(flat[:, s:s + cnt])
        s += cnt
    return out


def reconstruct_rotated(idx, d, bits1, bits2):
    """y_hat (unit norm) from the codes: the inverse recursion of the centroid angles."""
    cent = [codebook(l, w)[0][k] for l, (w, k) in enumerate(zip(level_bits(d, bits1, bits2), idx), start=1)]
    return unpolar(cent)


def key_logits(qprime, idx, norm16, d, bits1, bits2):
    """l_t = n_t <q', y_hat_t> for each query row of qprime [G, d] (or [d])."""
    y_hat = reconstruct_rotated(idx, d, bits1, bits2)
    return (np.atleast_2d(qprime) @ y_hat.T) * np.asarray(norm16)[None, :]


def decode(q, kcache, vcache, seq_lens, pi, bits1, bits2, v_centroids, scale=None, gqa_map=None):
    """Decode attention over PolarQuant keys and MSE values.

    q [B, Hq, d]; kcache: 'packed' [B, Hkv, T, stride] angle streams and
    'norm16' [B, Hkv, T]; vcache: 'idx' [B, Hkv, T, d] and 'norm16'.
    Returns (out [B, Hq, d], logits [B][Hq] -> [L_b])."""
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    hkv = kcache["norm16"].shape[1]
    if gqa_map is None:
        gqa_map = attention.default_gqa_map(hq, hkv)
    if scale is None or scale == 0:
        scale = 1.0 / np.sqrt(d)
    pi = np.asarray(pi, dtype=np.float64)
    out = np.zeros((bsz, hq, d))
    logits = [[None] * hq for _ in range(bsz)]
    for b in range(bsz):
        L = int(seq_lens[b])
        for h in range(hq):
            kv = int(gqa_map[h])
            if L == 0:
                continue  # no visible token: output 0
            qp = pi @ q[b, h]
            idx = unpack(kcache["packed"][b, kv, :L], d, bits1, bits2)
            l = key_logits(qp, idx, kcache["norm16"][b, kv, :L], d, bits1, bits2)[0]
            s = scale * l
            p = np.exp(s - np.max(s))
            p = p / np.sum(p)
            vhat = vcache["norm16"][b, kv, :L, None] * np.asarray(v_centroids)[vcache["idx"][b, kv, :L]]
            out[b, h] = (p @ vhat) @ pi
            logits[b][h] = l
    return out, logits
