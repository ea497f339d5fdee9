"""Pins for the oracle's quantize-on-append and packed layout (CPU only)."""

import json
import os

import numpy as np
import pytest

from conftest import GOLDEN
from oracle import attention, codebook, footprint, quantize, rng, rotation


def test_fp16_rne_matches_numpy_on_float32_inputs():
    x = rng.normals(2, 50000) * np.exp(rng.normals(3, 50000) * 3)
    x = x.astype(np.float32).astype(np.float64)
    mids = np.array([1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11, 2048.0 + 1.0, 2.0**-24 * 1.5, 2.0**-25, 65519.0])
    x = np.concatenate([x, mids, -mids])
    x = x[np.abs(x) <= 65504.0]
    want = x.astype(np.float32).astype(np.float16).astype(np.float64)
    assert np.array_equal(quantize.fp16_rne(x), want)


def test_fp16_saturates():
    assert quantize.fp16_rne(np.array([1e6, -7e4, 65504.0]))[:].tolist() == [65504.0, -65504.0, 65504.0]


def test_packing_golden_example():
    cases = json.load(open(os.path.join(GOLDEN, "packing_example.json")))["cases"]
    for c in cases:
        got = quantize.pack_codes(np.array([c["idx"]]), c["bprime"])[0].tobytes()
        assert got == bytes.fromhex(c["bytes_hex"].replace(" ", ""))


@pytest.mark.parametrize("d", [128, 200])
@pytest.mark.parametrize("bprime", [1, 2, 3, 4])
def test_pack_round_trip_and_padding(d, bprime):
    idx = np.random.default_rng(bprime).integers(0, 2**bprime, size=(5, d))
    p = quantize.pack_codes(idx, bprime)
    assert p.shape[1] % 16 == 0 and p.shape[1] == quantize.row_stride(bprime * d)
    assert np.array_equal(quantize.unpack_codes(p, d, bprime), idx)
    used = (bprime * d + 7) // 8
    assert np.all(p[:, used:] == 0)
    if (bprime * d) % 8:
        assert np.all(p[:, used - 1] >> ((bprime * d) % 8) == 0)
    z = np.random.default_rng(1).random((5, d)) < 0.5
    assert np.array_equal(quantize.unpack_signs(quantize.pack_signs(z), d), z)


def _unit_rows(n, d, seed):
    x = np.random.default_rng(seed).standard_normal((n, d))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


@pytest.mark.parametrize("bits", [2, 3])
def test_per_coordinate_mse_equals_distortion(bits):
    """Rotated unit vectors are uniform on the sphere, so E[(y_i - c[idx_i])^2] = D_b."""
    d, n = 128, 20000
    pi = rotation.dense_rotation(1, d)
    qz = quantize.quantize(_unit_rows(n, d, 4), pi, "mse", bits)
    err = ((qz["y"] - qz["centroids"][qz["idx"]]) ** 2).ravel()
    want = codebook.distortion(d, bits)
    assert abs(err.mean() - want) < 4 * err.std() / np.sqrt(err.size)


def test_cosine_at_three_bits_matches_printed_figure():
    """E cos(x, x~) = sqrt(1 - d D_3) = 0.9829 at d = 128, which the A2A page rounds to 0.983."""
    fig = json.load(open(os.path.join(GOLDEN, "page_figures.json")))["cosine_3bit"]["min_value"]
    d, n = 128, 5000
    pi = rotation.dense_rotation(1, d)
    x = _unit_rows(n, d, 5)
    qz = quantize.quantize(x, pi, "mse", 3)
    xt = quantize.reconstruct(qz, pi, "mse", use_stored_norms=False)
    cos = np.sum(x * xt, axis=1) / np.linalg.norm(xt, axis=1)
    theory = np.sqrt(1 - d * codebook.distortion(d, 3))
    assert abs(cos.mean() - theory) < 4 * cos.std() / np.sqrt(n) + 1e-4
    assert round(theory, 3) == fig


def _estimates(q, k, d, bits, seeds, mode, bits2=None):
    out = np.empty(seeds)
    for s in range(seeds):
        pi = rotation.dense_rotation(10_000 + s, d)
        smat = rng.round_to_bf16(rng.normals(90_000 + s, d * d).reshape(d, d)) if mode == "prod" else None
        qz = quantize.quantize(k[None], pi, mode, bits, smat, bits2=bits2)
        qp, u = attention.query_prep(q, pi, smat)
        c = qz["centroids"]
        if mode == "prod":
            out[s] = attention.key_logits(qp, u, qz["idx"], qz["n"], c, qz["gamma"], qz["z"], d)[0]
        else:
            out[s] = attention.key_logits(qp, None, qz["idx"], qz["n"], c)[0]
    return out


def test_prod_inner_product_is_unbiased_and_mse_is_not():
    """Over rotation/projection seeds the PROD estimate averages to <q,k>.

    The 1-bit MSE estimate instead averages to d c_1^2 <q,k> (c_1 the 1-bit
    centroid, d c_1^2 -> 2/pi): the bias the QJL stage exists to remove.
    """
    d, seeds = 32, 6000
    r = np.random.default_rng(0)
    k = r.standard_normal(d) * 3
    q = 0.8 * k / np.linalg.norm(k) * 2 + 0.6 * r.standard_normal(d)
    exact = q @ k
    est = _estimates(q, k, d, 2, seeds, "prod")
    se = est.std() / np.sqrt(seeds)
    assert abs(est.mean() - exact) < 3.5 * se
    mse = _estimates(q, k, d, 1, 2000, "mse")
    c1 = codebook.lloyd_max(d, 1)[0][1]
    se_m = mse.std() / np.sqrt(mse.size)
    assert abs(mse.mean() - d * c1 * c1 * exact) < 4 * se_m + 1e-9 * abs(exact)
    assert abs(mse.mean() - exact) > 10 * se_m


def test_gaussian_sign_identity():
    """E[sign(<s,r>) <s,y>] = sqrt(2/pi) <r,y>/||r|| for s ~ N(0, I): the QJL scale."""
    d, n = 16, 400_000
    r_ = np.random.default_rng(3)
    rv, yv = r_.standard_normal(d), r_.standard_normal(d)
    s = r_.standard_normal((n, d))
    vals = np.sign(s @ rv) * (s @ yv)
    want = np.sqrt(2 / np.pi) * (rv @ yv) / np.linalg.norm(rv)
    assert abs(vals.mean() - want) < 4 * vals.std() / np.sqrt(n)
    assert abs(quantize.qjl_scale(d) * d - np.sqrt(np.pi / 2)) < 1e-15


def test_estimator_equals_dense_reconstruction():
    d, n = 64, 50
    pi = rotation.dense_rotation(1, d)
    smat = rng.round_to_bf16(rng.normals(2, d * d).reshape(d, d))
    x = np.random.default_rng(6).standard_normal((n, d)) * 5
    q = np.random.default_rng(7).standard_normal(d)
    qz = quantize.quantize(x, pi, "prod", 3, smat)
    qp, u = attention.query_prep(q, pi, smat)
    l = attention.key_logits(qp, u, qz["idx"], qz["norm16"], qz["centroids"], qz["rnorm16"], qz["z"], d)
    xt = quantize.reconstruct(qz, pi, "prod", smat)
    assert np.max(np.abs(l - xt @ q)) < 1e-10 * np.max(np.abs(l))


def test_zero_vector():
    d = 128
    pi = rotation.dense_rotation(1, d)
    smat = rng.round_to_bf16(rng.normals(2, d * d).reshape(d, d))
    qz = quantize.quantize(np.zeros((1, d)), pi, "prod", 3, smat)
    assert qz["norm16"][0] == 0.0
    assert np.all(qz["idx"] == 2)  # y = 0 sits on the middle boundary, upper cell
    c = qz["centroids"]
    assert abs(qz["gamma"][0] - abs(c[2]) * np.sqrt(d)) < 1e-15


def test_footprint_matches_printed_turbo_figures():
    figs = json.load(open(os.path.join(GOLDEN, "page_figures.json")))
    assert footprint.bytes_per_vector("prod", 3, 128) == 52
    assert footprint.bits_per_value("prod", 3, 128) == figs["turbo3"]["bits_per_value"]
    assert footprint.bits_per_value("prod", 4, 128) == figs["turbo4"]["bits_per_value"]
    assert round(footprint.ratio_vs_fp16("prod", 3, 128), 1) == figs["turbo3"]["ratio_vs_fp16"]
    assert round(footprint.ratio_vs_fp16("prod", 4, 128), 1) == figs["turbo4"]["ratio_vs_fp16"]
    ctx = figs["context_70b_34gb"]
    assert abs(ctx["fp16_tokens"] * footprint.ratio_vs_fp16("prod", 3, 128) / ctx["tq3_tokens"] - 1) < 0.01
    assert footprint.bytes_per_vector("mse", 3, 128) == 50
    assert footprint.bytes_per_vector("prod", 3, 200, padded=True) == 64 + 32 + 4
    assert footprint.bytes_per_vector("prod", 2, 200, padded=True) == 32 + 32 + 4


# ---- fractional bit-rates: two channel groups (i mod 16 < 8 at `bits`, the rest at `bits2`) ----

@pytest.mark.parametrize("mode,bits", [("mse", 3), ("prod", 3), ("prod", 4)])
def test_two_groups_of_equal_width_are_the_single_width_quantizer(mode, bits):
    d = 128
    pi = rotation.dense_rotation(1, d)
    smat = rng.round_to_bf16(rng.normals(2, d * d).reshape(d, d)) if mode == "prod" else None
    x = np.random.default_rng(8).standard_normal((40, d))
    a = quantize.quantize(x, pi, mode, bits, smat)
    b = quantize.quantize(x, pi, mode, bits, smat, bits2=bits)
    assert np.array_equal(a["idx"], b["idx"])
    assert np.array_equal(quantize.pack(a, mode, bits)["codes"], quantize.pack(b, mode, bits, bits)["codes"])


def test_two_group_packing_by_hand():
    """d = 16, widths 2 (coordinates 0..7) and 1 (8..15), LSB first: codes
    3,0,1,2,3,0,1,2 give bit pairs 11 00 10 01 -> 0b10010011 = 0x93 twice;
    codes 1,0,1,1,0,0,1,0 give 0b01001101 = 0x4d; a two-width row is padded
    to 8 bytes (not 16), so the narrower group saves memory."""
    idx = np.array([[3, 0, 1, 2, 3, 0, 1, 2, 1, 0, 1, 1, 0, 0, 1, 0]])
    w = quantize.code_widths(16, "prod", 3, 2)
    assert w.tolist() == [2] * 8 + [1] * 8
    got = quantize.pack_codes(idx, w)
    assert got[0].tobytes() == bytes([0x93, 0x93, 0x4D] + [0] * 5)
    assert np.array_equal(quantize.unpack_codes(got, 16, w), idx)


@pytest.mark.parametrize("bits,bits2", [(3, 2), (4, 3)])
def test_two_group_mse_per_group_equals_each_distortion(bits, bits2):
    """Each group is quantized with its own Lloyd-Max codebook of the same
    Beta law: per coordinate E[(y_i - c[idx_i])^2] = D_bits on the first
    group and D_bits2 on the second."""
    d, n = 128, 20000
    pi = rotation.dense_rotation(1, d)
    qz = quantize.quantize(_unit_rows(n, d, 9), pi, "mse", bits, bits2=bits2)
    err = (qz["y"] - quantize.coord_centroids(qz["centroids"], qz["idx"])) ** 2
    first = quantize.in_first_group(d)
    for sel, b in ((first, bits), (~first, bits2)):
        e = err[:, sel].ravel()
        assert abs(e.mean() - codebook.distortion(d, b)) < 4 * e.std() / np.sqrt(e.size)


def test_two_group_prod_inner_product_is_unbiased():
    """Keys at 2.5 bits (3 / 2): the estimate still averages to <q,k> over seeds."""
    d, seeds = 32, 3000
    r = np.random.default_rng(1)
    k = r.standard_normal(d) * 3
    q = 0.8 * k / np.linalg.norm(k) * 2 + 0.6 * r.standard_normal(d)
    est = _estimates(q, k, d, 3, seeds, "prod", bits2=2)
    assert abs(est.mean() - q @ k) < 3.5 * est.std() / np.sqrt(seeds)


def test_two_group_estimator_equals_dense_reconstruction():
    d, n = 64, 50
    pi = rotation.dense_rotation(1, d)
    smat = rng.round_to_bf16(rng.normals(2, d * d).reshape(d, d))
    x = np.random.default_rng(6).standard_normal((n, d)) * 5
    q = np.random.default_rng(7).standard_normal(d)
    qz = quantize.quantize(x, pi, "prod", 4, smat, bits2=3)
    qp, u = attention.query_prep(q, pi, smat)
    l = attention.key_logits(qp, u, qz["idx"], qz["norm16"], qz["centroids"], qz["rnorm16"], qz["z"], d)
    xt = quantize.reconstruct(qz, pi, "prod", smat)
    assert np.max(np.abs(l - xt @ q)) < 1e-10 * np.max(np.abs(l))


def test_two_group_footprint():
    """2.5 and 3.5 bits per channel: keys 1.5 / 2.5 code bits + 1 sign bit per
    coordinate plus two float16 scalars per 128 coordinates."""
    assert footprint.bytes_per_vector("prod", 3, 128, bits2=2) == 24 + 16 + 4
    assert footprint.bits_per_value("prod", 3, 128, bits2=2) == 2.75
    assert footprint.bytes_per_vector("prod", 4, 128, bits2=3) == 40 + 16 + 4
    assert footprint.bits_per_value("prod", 4, 128, bits2=3) == 3.75
    assert footprint.bytes_per_vector("mse", 3, 128, bits2=2) == 40 + 2
