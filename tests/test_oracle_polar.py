"""Pins of the PolarQuant oracle (oracle/polar.py) against what the pages and
the mathematics fix: the exact inverse of the polar recursion, the angle laws
after a Haar rotation, the Lloyd-Max conditions of every level's codebook
(checked with an independent adaptive quadrature and with Monte Carlo), the
closed-form distortion of one uniform angle (d = 2), logits equal to the dense
reconstruction's dot products, and a hand-worked packing example."""

import json
import os

import numpy as np
import pytest
from scipy import integrate, stats

from oracle import polar as P
from oracle import rotation as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _haar_unit(n, d, seed):
    g = np.random.default_rng(seed).standard_normal((n, d))
    return g / np.linalg.norm(g, axis=1, keepdims=True)


@pytest.mark.parametrize("d", [2, 4, 16, 128])
def test_polar_inverse_is_exact(d):
    y = np.random.default_rng(d).standard_normal((300, d)) * np.random.default_rng(d + 1).lognormal(0, 2, (300, 1))
    ang, rad = P.polar(y)
    assert len(ang) == P.levels(d) and [a.shape[1] for a in ang] == P.angle_count(d)
    assert np.allclose(rad, np.linalg.norm(y, axis=1), rtol=1e-14, atol=0)
    back = P.unpolar(ang, rad)
    assert np.max(np.abs(back - y) / np.max(np.abs(y), axis=1, keepdims=True)) < 1e-14
    # level 1 angles live on the circle, higher levels in the first quadrant
    assert np.all(np.abs(ang[0]) <= np.pi)
    for a in ang[1:]:
        assert np.all((a >= 0) & (a <= np.pi / 2))


def test_angle_laws_after_haar_rotation():
    """Level 1 uniform on the circle; level l >= 2: sin^2 psi ~ Beta(k/2, k/2),
    k = 2^(l-1). A wrong exponent or block size fails the KS test."""
    y = _haar_unit(6000, 128, 7)
    ang, _ = P.polar(y)
    for l in range(1, 8):
        a = ang[l - 1].ravel()
        p = stats.kstest(a, lambda v: P.angle_cdf(v, l)).pvalue
        assert p > 1e-4, f"level {l}: KS p = {p}"
        if l >= 2:  # the neighbouring law (k off by a factor 2) is rejected
            wrong = stats.kstest(a, lambda v: P.angle_cdf(v, l + 1)).pvalue
            assert wrong < 1e-6, f"level {l}: the law of level {l + 1} fits too ({wrong})"


@pytest.mark.parametrize("level", [2, 3, 5, 7])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_codebook_lloyd_max_conditions(level, bits):
    """Boundaries are midpoints; each centroid is the conditional mean of its
    cell, recomputed here with scipy's adaptive quadrature (not the oracle's
    Gauss-Legendre with the incomplete-beta mass); symmetric about pi/4."""
    c, t = P.codebook(level, bits)
    assert np.all(np.diff(c) > 0) and len(c) == 1 << bits
    assert np.allclose(t, 0.5 * (c[:-1] + c[1:]), rtol=0, atol=1e-15)
    assert np.allclose(c + c[::-1], np.pi / 2, rtol=0, atol=1e-13)
    edges = np.concatenate(([0.0], t, [np.pi / 2]))
    for i in range(len(c)):
        f = lambda u: float(P.angle_pdf(u, level))  # noqa: E731
        mass = integrate.quad(f, edges[i], edges[i + 1], epsabs=1e-14, epsrel=1e-12, limit=400)[0]
        mom = integrate.quad(lambda u: u * f(u), edges[i], edges[i + 1], epsabs=1e-14, epsrel=1e-12, limit=400)[0]
        assert abs(mom / mass - c[i]) < 1e-9, (level, bits, i, mom / mass, c[i])


def test_level1_codebook_is_the_uniform_grid():
    for bits in (1, 2, 3, 4):
        c, t = P.codebook(1, bits)
        w = 2 * np.pi / (1 << bits)
        assert np.allclose(c, -np.pi + w * (np.arange(1 << bits) + 0.5), atol=1e-15)
        assert np.allclose(t, -np.pi + w * np.arange(1, 1 << bits), atol=1e-15)


def test_codebook_centroids_match_monte_carlo_and_are_optimal():
    """Empirical conditional means of the angles of Haar-random vectors match
    the centroids within 3 standard errors, and moving the centroids off the
    fixed point raises the empirical distortion."""
    y = _haar_unit(20000, 64, 11)
    ang, _ = P.polar(y)
    for level, bits in ((2, 2), (4, 2), (6, 3)):
        a = ang[level - 1].ravel()
        c, t = P.codebook(level, bits)
        k = np.searchsorted(t, a, side="right")
        for i in range(len(c)):
            sel = a[k == i]
            se = sel.std() / np.sqrt(sel.size)
            assert abs(sel.mean() - c[i]) < 3 * se + 1e-12, (level, bits, i)
        base = np.mean((a - c[k]) ** 2)
        for eps in (0.02, -0.02):
            moved = c + eps * (np.arange(len(c)) - (len(c) - 1) / 2) / len(c)
            assert np.mean((a - moved[k]) ** 2) > base


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_one_uniform_angle_closed_form_distortion(bits):
    """d = 2: the only angle is uniform and its quantizer has equal cells of
    width w, so E||y - y_hat||^2 = 2 - 2 sin(w/2) / (w/2) for a unit y."""
    y = _haar_unit(200000, 2, 3 + bits)
    qz = P.quantize(y, np.eye(2), bits1=bits, bits2=bits)
    err = np.sum((qz["y"] - qz["y_hat"]) ** 2, axis=1)
    w = 2 * np.pi / (1 << bits)
    want = 2.0 - 2.0 * np.sin(w / 2) / (w / 2)
    assert abs(err.mean() - want) < 3 * err.std() / np.sqrt(err.size)


def test_reconstruction_unit_norm_and_quality():
    """y_hat has unit norm exactly; at 4 / 2 bits (382 bits per 128-vector) the
    mean cosine to the rotated input is close to the MSE codebook's 3-bit
    figure (a quality report, loosely bounded)."""
    x = np.random.default_rng(5).standard_normal((500, 128))
    pi = R.make_rotation(1, 128, "dense")
    qz = P.quantize(x, pi, 4, 2)
    assert np.allclose(np.linalg.norm(qz["y_hat"], axis=1), 1.0, atol=1e-14)
    assert P.row_bits(128, 4, 2) == 64 * 4 + 63 * 2
    cos = np.sum(qz["y"] * qz["y_hat"], axis=1)
    assert 0.97 < cos.mean() < 0.995


def test_key_logits_equal_dense_reconstruction():
    """n <q', y_hat> equals <q, n Pi^T y_hat> (the key rebuilt in the input space)."""
    d = 128
    for kind in ("dense", "rht"):
        pi = R.make_rotation(1, d, kind)
        x = np.random.default_rng(2).standard_normal((64, d)) * 3
        q = np.random.default_rng(3).standard_normal((4, d))
        qz = P.quantize(x, pi, 4, 2)
        got = P.key_logits(R.rotate(pi, q), qz["idx"], qz["norm16"], d, 4, 2)
        khat = qz["norm16"][:, None] * R.unrotate(pi, qz["y_hat"])
        assert np.allclose(got, q @ khat.T, rtol=1e-12, atol=1e-12)


def test_packing_hand_worked_example():
    """d = 4, bits 3 / 2: level-1 codes (5, 2) and the level-2 code 1 give
    stream bits 1,0,1, 0,1,0, 1,0 (LSB first): byte 0 = 0x55 and nothing else,
    worked out by hand in tests/golden/polar_packing_example.json."""
    with open(os.path.join(GOLDEN, "polar_packing_example.json")) as f:
        g = json.load(f)
    idx = [np.array([g["level1"]]), np.array([[g["level2"]]])]
    packed = P.pack(idx, 4, g["bits1"], g["bits2"])
    assert packed.shape == (1, 16)
    assert packed[0, :2].tolist() == g["bytes"] and not packed[0, 2:].any()
    back = P.unpack(packed, 4, g["bits1"], g["bits2"])
    assert back[0].tolist() == [g["level1"]] and back[1].tolist() == [[g["level2"]]]
    # random round trip at d = 128
    rng = np.random.default_rng(0)
    idx = [rng.integers(0, 1 << w, (10, cnt)) for cnt, w in zip(P.angle_count(128), P.level_bits(128, 4, 2))]
    back = P.unpack(P.pack(idx, 128, 4, 2), 128, 4, 2)
    assert all(np.array_equal(a, b) for a, b in zip(idx, back))


def test_decode_is_softmax_attention_over_reconstructions():
    """polar.decode equals the generic rotated-domain attention (textbook
    softmax over <q', khat_t>, value sum, un-rotation) fed the explicit key
    reconstructions n_t y_hat_t, for two batches, GQA 2 and a ragged length."""
    from oracle import attention as A
    from oracle import codebook as C
    d, bsz, hkv, T = 128, 2, 2, 40
    rng = np.random.default_rng(9)
    pi = R.make_rotation(4, d, "rht")
    k = rng.standard_normal((bsz, hkv, T, d)) * 2
    v = rng.standard_normal((bsz, hkv, T, d))
    q = rng.standard_normal((bsz, 4, d))
    qz = P.quantize(k.reshape(-1, d), pi, 4, 2)
    packed = P.pack(qz["idx"], d, 4, 2).reshape(bsz, hkv, T, -1)
    vc, vt = C.lloyd_max(d, 3)
    vy = (v.reshape(-1, d) @ pi.T) / np.linalg.norm(v.reshape(-1, d), axis=1, keepdims=True)
    vidx = np.searchsorted(vt, vy, side="right").reshape(bsz, hkv, T, d)
    vn = np.linalg.norm(v, axis=-1)
    kcache = {"packed": packed, "norm16": qz["norm16"].reshape(bsz, hkv, T)}
    vcache = {"idx": vidx, "norm16": vn}
    lens = [T, 17]
    out, logits = P.decode(q, kcache, vcache, lens, pi, 4, 2, vc)
    yhat = P.reconstruct_rotated(qz["idx"], d, 4, 2).reshape(bsz, hkv, T, d)
    for b in range(bsz):
        for h in range(4):
            kv = h // 2
            L = lens[b]
            khat = kcache["norm16"][b, kv, :L, None] * yhat[b, kv, :L]
            vhat = vn[b, kv, :L, None] * vc[vidx[b, kv, :L]]
            want, wl = A.attention_from_rotated(pi @ q[b, h], khat, vhat, 1 / np.sqrt(d), pi)
            assert np.allclose(out[b, h], want, rtol=1e-12, atol=1e-12)
            assert np.allclose(logits[b][h], wl, rtol=1e-12, atol=1e-12)
