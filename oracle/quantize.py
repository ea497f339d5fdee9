"""Quantize-on-append, fp64 oracle: norm, rotate, bucketize, pack, residual QJL.

What the write-ups say:
* the vector is normalised and its norm kept aside (A2A TurboQuant explainer,
  section "Stage 1", first bullet under PolarQuant);
* it is rotated by the fixed random orthogonal matrix and each coordinate is
  mapped to a low-bit index by the Lloyd-Max quantizer of the Beta law
  (same section; Qiita TurboQuant article, "Rotate, then quantize");
* the two-stage variant rounds with the MSE quantizer first and then applies a
  1-bit Quantized Johnson-Lindenstrauss transform to the residual so the
  inner-product estimate becomes unbiased (Qiita, "One more stage so attention
  does not break"; A2A, "Stage 2: QJL residual correction");
* attention is then scored straight from the stored indices (A2A, end of
  "Stage 2").

Readings (the pages are silent or garbled):
* MSE mode (values) uses b bits per coordinate; PROD mode (keys) uses b-1 bits
  of Lloyd-Max plus m sign bits of S r, m = d unless stated (A2A "Stage 2"
  says "1 bit per vector ... +1 or 5"; read as one sign bit per projected
  coordinate, +1 or -1);
* S is m x d, standard normal draws rounded to bfloat16, applied to the
  residual in the rotated domain, r = y - c[idx] with y = Pi x / ||x||;
* the norms ||x|| and gamma = ||r|| are stored as float16, round to nearest
  even, saturated at 65504;
* a zero vector gets n = 0 and y = 0 and then goes through the same steps;
* a coordinate equal to a boundary goes to the upper cell.

Fractional bit-rates (2.5 / 3.5 bits per channel, Qiita "Which bit-width is
lossless" and A2A "Benchmarks and real-world performance" quote them; the
mechanism is not on the pages): the plainest reading, two groups of channels
at different bit widths, each with its own Lloyd-Max codebook of the same Beta
law. After the rotation every coordinate has that law, so which coordinates
carry the extra bit is free; this project puts coordinate i in the first group
(`bits`) when i mod 16 < 8 and in the second (`bits2`) otherwise, and packs
the codes in coordinate order, each with its own width. 2.5 bits = b 3 / 2,
3.5 = 4 / 3 (for keys, b counts the sign bit: code widths b - 1).

Packed layout (this project's specification; the pages give none):
* codes: LSB-first bit stream, bit k of coordinate i's index at stream bit
  o_i + k with o_i the sum of the widths of coordinates 0 .. i-1 (b'*i for one
  width), stream bit p in byte p // 8 at bit p % 8; row stride = the byte
  count rounded up to 16 (to 8 with two widths, so the narrower group saves
  memory); padding bits 0;
* signs: bit j = [(S r)_j >= 0] at byte j // 8, bit j % 8; stride rounded up
  to 16;
* norm / rnorm: float16 per vector.

Pinned by: per-coordinate MSE equal to the codebook's distortion, the cosine
figure the A2A page prints for 3 bits, the unbiasedness of the PROD inner
product over seeds (and the 2/pi bias of 1-bit MSE without it), a hand-worked
packing example (tests/golden/packing_example.json); the exact byte layout
itself is this project's spec (parity unpinned beyond that example and the
round trip).
"""

import numpy as np

from . import codebook, rotation


def fp16_rne(x):
    """Round float64 to the nearest float16 (ties to even), saturating at 65504.

    Returned as float64 holding the float16 value.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), 65504.0)
    out = np.empty_like(a)
    small = a < 2.0**-14
    out[small] = np.rint(a[small] * 2.0**24) * 2.0**-24  # subnormal spacing
    m, e = np.frexp(a[~small])
    out[~small] = np.ldexp(np.rint(m * 2048.0), e - 11)  # 11 significant bits
    out = np.minimum(out, 65504.0)
    return np.copysign(out, x)


def code_bits(mode, bits):
    """Lloyd-Max bits per coordinate: b for MSE (values), b-1 for PROD (keys)."""
    if mode == "mse":
        if not 1 <= bits <= 4:
            raise ValueError("MSE bits must be 1..4")
        return bits
    if mode == "prod":
        if not 2 <= bits <= 5:
            raise ValueError("PROD bits must be 2..5")
        return bits - 1
    raise ValueError(mode)


def row_stride(nbits_per_row):
    nbytes = (nbits_per_row + 7) // 8
    return (nbytes + 15) // 16 * 16


def in_first_group(d):
    """bool [d]: coordinate i takes the first width (i mod 16 < 8)."""
    return (np.arange(d) % 16) < 8


def code_widths(d, mode, bits, bits2=None):
    """Code bits of each coordinate: one width, or the two groups' widths."""
    bp = code_bits(mode, bits)
    if bits2 is None or bits2 == bits:
        return np.full(d, bp, dtype=np.int64)
    return np.where(in_first_group(d), bp, code_bits(mode, bits2)).astype(np.int64)


def coord_centroids(centroids, idx):
    """The centroid value of every code: centroids is one table [L] or one
    table per coordinate [d, L] (two-group caches); idx [..., d]."""
    c = np.asarray(centroids)
    if c.ndim == 1:
        return c[idx]
    return c[np.arange(c.shape[0]), idx]


def quantize(x, pi, mode, bits, s_matrix=None, bits2=None):
    """Quantize rows of x (float64 [n, d]); bits2: the second group's bits of
    a fractional-rate cache (None: every coordinate at `bits`).

    Returns a dict with: n (exact norm), norm16, y (rotated unit vector), idx
    (codes, int64 [n, d]), centroids ([L], or [d, L] with each coordinate's
    table when there are two groups), boundaries (likewise), widths; for PROD
    also r, gamma, rnorm16, sproj (= S r) and z (bool [n, m]).
    """
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    d = x.shape[1]
    bp = code_bits(mode, bits)
    c, t = codebook.lloyd_max(d, bp)
    n = np.sqrt(np.sum(x * x, axis=1))
    safe = np.where(n > 0, n, 1.0)
    y = rotation.rotate(pi, x) / safe[:, None]
    y[n == 0] = 0.0
    widths = code_widths(d, mode, bits, bits2)
    if np.all(widths == bp):
        idx = codebook.bucketize(y, t)
    else:
        # each group bucketized with its own codebook; tables padded to a common length
        c2, t2 = codebook.lloyd_max(d, code_bits(mode, bits2))
        first = in_first_group(d)
        idx = np.where(first, codebook.bucketize(y, t), codebook.bucketize(y, t2))
        lmax = max(len(c), len(c2))
        ctab = np.full((d, lmax), np.nan)
        ttab = np.full((d, lmax - 1), np.nan)
        ctab[first, : len(c)] = c
        ctab[~first, : len(c2)] = c2
        ttab[first, : len(t)] = t
        ttab[~first, : len(t2)] = t2
        c, t = ctab, ttab
    out = {"n": n, "norm16": fp16_rne(n), "y": y, "idx": idx, "centroids": c, "boundaries": t, "widths": widths}
    if mode == "prod":
        if s_matrix is None:
            raise ValueError("PROD mode needs the QJL matrix S")
        r = y - coord_centroids(c, idx)
        gamma = np.sqrt(np.sum(r * r, axis=1))
        sproj = r @ np.asarray(s_matrix, dtype=np.float64).T
        out.update(r=r, gamma=gamma, rnorm16=fp16_rne(gamma), sproj=sproj, z=sproj >= 0.0)
    return out


def _widths(d, bprime):
    w = np.asarray(bprime, dtype=np.int64)
    return np.full(d, int(w), dtype=np.int64) if w.ndim == 0 else w


def pack_codes(idx, bprime):
    """LSB-first bit stream per row; bprime is one width (stride rounded up to
    16 bytes) or the width of every coordinate (two widths: stride rounded up
    to 8 bytes)."""
    idx = np.atleast_2d(np.asarray(idx, dtype=np.int64))
    n, d = idx.shape
    w = _widths(d, bprime)
    off = np.concatenate([[0], np.cumsum(w)])
    if np.all(w == w[0]):
        stride = row_stride(int(off[-1]))
    else:
        stride = ((int(off[-1]) + 7) // 8 + 7) // 8 * 8
    out = np.zeros((n, stride), dtype=np.uint8)
    for i in range(d):
        for k in range(int(w[i])):
            p = int(off[i]) + k
            bit = ((idx[:, i] >> k) & 1).astype(np.uint8)
            out[:, p // 8] |= bit << np.uint8(p % 8)
    return out


def unpack_codes(packed, d, bprime):
    packed = np.atleast_2d(np.asarray(packed, dtype=np.uint8))
    w = _widths(d, bprime)
    off = np.concatenate([[0], np.cumsum(w)])
    idx = np.zeros((packed.shape[0], d), dtype=np.int64)
    for i in range(d):
        for k in range(int(w[i])):
            p = int(off[i]) + k
            bit = (packed[:, p // 8] >> np.uint8(p % 8)) & 1
            idx[:, i] |= bit.astype(np.int64) << k
    return idx


def pack_signs(z):
    z = np.atleast_2d(np.asarray(z, dtype=bool))
    n, m = z.shape
    out = np.zeros((n, row_stride(m)), dtype=np.uint8)
    for j in range(m):
        out[:, j // 8] |= z[:, j].astype(np.uint8) << np.uint8(j % 8)
    return out


def unpack_signs(packed, m):
    packed = np.atleast_2d(np.asarray(packed, dtype=np.uint8))
    z = np.zeros((packed.shape[0], m), dtype=bool)
    for j in range(m):
        z[:, j] = ((packed[:, j // 8] >> np.uint8(j % 8)) & 1) == 1
    return z


def pack(qz, mode, bits, bits2=None):
    """Packed planes of one quantize() result: codes, signs (PROD), norm, rnorm (PROD)."""
    d = qz["idx"].shape[1]
    planes = {
        "codes": pack_codes(qz["idx"], code_widths(d, mode, bits, bits2)),
        "norm": qz["norm16"].astype(np.float16),
    }
    if mode == "prod":
        planes["signs"] = pack_signs(qz["z"])
        planes["rnorm"] = qz["rnorm16"].astype(np.float16)
    planes["d"] = d
    return planes


def qjl_scale(m):
    """sqrt(pi/2) / m: E|g| = sqrt(2/pi) for g ~ N(0,1) makes the sign sketch unbiased."""
    return np.sqrt(np.pi / 2.0) / m


def reconstruct(qz, pi, mode, s_matrix=None, use_stored_norms=True):
    """Explicit dense reconstruction x~ (used only to pin the logit estimator).

    MSE:  x~ = n Pi^T c[idx]
    PROD: x~ = n Pi^T (c[idx] + sqrt(pi/2)/m * gamma * S^T (2z - 1))
    """
    n = qz["norm16"] if use_stored_norms else qz["n"]
    yhat = coord_centroids(qz["centroids"], qz["idx"])
    if mode == "prod":
        s = np.asarray(s_matrix, dtype=np.float64)
        g = qz["rnorm16"] if use_stored_norms else qz["gamma"]
        pm = 2.0 * qz["z"].astype(np.float64) - 1.0
        yhat = yhat + qjl_scale(s.shape[0]) * g[:, None] * (pm @ s)
    return n[:, None] * rotation.unrotate(pi, yhat)
