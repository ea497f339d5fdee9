"""Pins for the oracle's decode attention and top-k search (CPU only)."""

import numpy as np

from oracle import attention, quantize, rng, rotation, topk


def _softmax_attention(q, k, v):
    """Textbook softmax(q K^T / sqrt(d)) V for one query row."""
    s = k @ q / np.sqrt(q.size)
    w = np.exp(s - s.max())
    return (w / w.sum()) @ v


def test_identity_quantizer_reduces_to_textbook_attention():
    d, t = 64, 37
    r = np.random.default_rng(0)
    q, k, v = r.standard_normal(d), r.standard_normal((t, d)) * 2, r.standard_normal((t, d))
    for kind in ("dense", "rht"):
        pi = rotation.make_rotation(1, d, kind)
        qp, _ = attention.query_prep(q, pi)
        out, logits = attention.attention_from_rotated(qp, rotation.rotate(pi, k), rotation.rotate(pi, v),
                                                       1 / np.sqrt(d), pi)
        assert np.max(np.abs(out - _softmax_attention(q, k, v))) < 1e-12
        assert np.max(np.abs(logits - k @ q)) < 1e-11


def _quantized_cache(b, hkv, t, d, seed, pi, smat, kbits, vbits):
    r = np.random.default_rng(seed)
    k = r.standard_normal((b, hkv, t, d)) * 3
    v = r.standard_normal((b, hkv, t, d))
    kq = quantize.quantize(k.reshape(-1, d), pi, "prod", kbits, smat)
    vq = quantize.quantize(v.reshape(-1, d), pi, "mse", vbits)
    sh = (b, hkv, t)
    kc = {"idx": kq["idx"].reshape(sh + (d,)), "norm16": kq["norm16"].reshape(sh),
          "rnorm16": kq["rnorm16"].reshape(sh), "z": kq["z"].reshape(sh + (d,))}
    vc = {"idx": vq["idx"].reshape(sh + (d,)), "norm16": vq["norm16"].reshape(sh)}
    return kq, vq, kc, vc


def test_decode_equals_generic_path_on_reconstructions():
    """decode() must equal softmax attention over the explicit reconstructions."""
    b, hq, hkv, t, d = 2, 4, 2, 19, 32
    pi = rotation.dense_rotation(1, d)
    smat = rng.round_to_bf16(rng.normals(2, d * d).reshape(d, d))
    kq, vq, kc, vc = _quantized_cache(b, hkv, t, d, 3, pi, smat, 3, 3)
    q = np.random.default_rng(4).standard_normal((b, hq, d))
    lens = np.array([t, 7])
    out, logits = attention.decode(q, kc, vc, lens, pi, smat, kq["centroids"], vq["centroids"])
    kt = quantize.reconstruct(kq, pi, "prod", smat).reshape(b, hkv, t, d)
    vt = quantize.reconstruct(vq, pi, "mse").reshape(b, hkv, t, d)
    for bi in range(b):
        for h in range(hq):
            kv = h // (hq // hkv)
            L = lens[bi]
            want = _softmax_attention(q[bi, h], kt[bi, kv, :L], vt[bi, kv, :L])
            assert np.max(np.abs(out[bi, h] - want)) < 1e-10
            assert np.max(np.abs(logits[bi][h] - kt[bi, kv, :L] @ q[bi, h])) < 1e-9


def test_single_token_returns_its_reconstruction_and_gqa_map():
    d = 16
    pi = rotation.rht_rotation(1, d)
    smat = rng.round_to_bf16(rng.normals(2, d * d).reshape(d, d))
    kq, vq, kc, vc = _quantized_cache(1, 2, 1, d, 5, pi, smat, 2, 4)
    q = np.random.default_rng(6).standard_normal((1, 6, d))
    out, _ = attention.decode(q, kc, vc, [1], pi, smat, kq["centroids"], vq["centroids"])
    vt = quantize.reconstruct(vq, pi, "mse").reshape(1, 2, 1, d)
    assert attention.default_gqa_map(6, 2).tolist() == [0, 0, 0, 1, 1, 1]
    for h in range(6):
        assert np.max(np.abs(out[0, h] - vt[0, h // 3, 0])) < 1e-12


def test_empty_sequence_gives_zero_output():
    d = 16
    pi = rotation.dense_rotation(1, d)
    smat = rng.round_to_bf16(rng.normals(2, d * d).reshape(d, d))
    kq, vq, kc, vc = _quantized_cache(1, 1, 3, d, 5, pi, smat, 3, 3)
    out, logits = attention.decode(np.ones((1, 2, d)), kc, vc, [0], pi, smat, kq["centroids"], vq["centroids"])
    assert np.all(out == 0)


def test_topk_brute_force_and_ties():
    s = np.array([[0.5, 2.0, 2.0, -1.0, 3.0, 2.0],
                  [1.0, 1.0, 1.0, 1.0, 1.0, 1.0]])
    ids, vals = topk.topk(s, 4)
    assert ids.tolist() == [[4, 1, 2, 5], [0, 1, 2, 3]]
    assert vals.tolist() == [[3.0, 2.0, 2.0, 2.0], [1.0, 1.0, 1.0, 1.0]]
    r = np.random.default_rng(1).standard_normal((3, 200))
    ids, _ = topk.topk(r, 10)
    for i in range(3):
        assert ids[i].tolist() == list(np.argsort(-r[i], kind="stable")[:10])


def test_search_scores_match_logit_estimator_and_recall_improves_with_bits():
    from online_kv_cache_quantize_gb300 import workloads
    d = 200
    db, qs = workloads.mixture_vectors(3000, d=d, queries=20)
    pi = rotation.dense_rotation(1, d)
    smat = rng.round_to_bf16(rng.normals(2, d * d).reshape(d, d))
    truth, _ = topk.exact_topk(qs, db, 10)
    rec = {}
    for bits in (2, 4):
        qz = quantize.quantize(db, pi, "prod", bits, smat)
        sc = topk.scores(qs, pi, smat, qz["idx"], qz["norm16"], qz["centroids"], qz["rnorm16"], qz["z"])
        xt = quantize.reconstruct(qz, pi, "prod", smat)
        assert np.max(np.abs(sc - qs.astype(np.float64) @ xt.T)) < 1e-9
        ids, _ = topk.topk(sc, 10)
        rec[bits] = topk.recall_at_k(ids, truth)
    assert rec[4] > rec[2] > 0.3


def _causal_attention(q, k, v, start):
    """Textbook causal attention for a chunk of queries at positions start,
    start+1, ...: softmax(Q K^T / sqrt(d) + M) V with M[i, t] = -inf for t > start + i."""
    c, d = q.shape
    s = q @ k.T / np.sqrt(d)
    mask = np.arange(k.shape[0])[None, :] <= (start + np.arange(c))[:, None]
    s = np.where(mask, s, -np.inf)
    w = np.exp(s - s.max(axis=1, keepdims=True))
    return (w / w.sum(axis=1, keepdims=True)) @ v


def test_prefill_equals_causal_attention_on_reconstructions():
    """prefill() = causal masked softmax attention (one matrix expression) over
    the explicit reconstructions, chunk starting mid-sequence, GQA 2, whole
    width and two-group caches."""
    bsz, c, hq, hkv, t, d = 2, 5, 4, 2, 23, 32
    pi = rotation.dense_rotation(1, d)
    smat = rng.round_to_bf16(rng.normals(2, d * d).reshape(d, d))
    r = np.random.default_rng(9)
    k = r.standard_normal((bsz, hkv, t, d)) * 3
    v = r.standard_normal((bsz, hkv, t, d))
    q = r.standard_normal((bsz, c, hq, d))
    start = np.array([11, 0])
    for bits2 in (None, 2):
        kq = quantize.quantize(k.reshape(-1, d), pi, "prod", 3, smat, bits2=bits2)
        vq = quantize.quantize(v.reshape(-1, d), pi, "mse", 3, bits2=bits2)
        sh = (bsz, hkv, t)
        kc = {"idx": kq["idx"].reshape(sh + (d,)), "norm16": kq["norm16"].reshape(sh),
              "rnorm16": kq["rnorm16"].reshape(sh), "z": kq["z"].reshape(sh + (d,))}
        vc = {"idx": vq["idx"].reshape(sh + (d,)), "norm16": vq["norm16"].reshape(sh)}
        out = attention.prefill(q, kc, vc, start, pi, smat, kq["centroids"], vq["centroids"])
        kt = quantize.reconstruct(kq, pi, "prod", smat).reshape(bsz, hkv, t, d)
        vt = quantize.reconstruct(vq, pi, "mse").reshape(bsz, hkv, t, d)
        for b in range(bsz):
            for h in range(hq):
                kv = h // (hq // hkv)
                want = _causal_attention(q[b, :, h], kt[b, kv], vt[b, kv], start[b])
                assert np.max(np.abs(out[b, :, h] - want)) < 1e-10, (bits2, b, h)


def test_prefill_of_one_token_is_decode():
    b, hq, hkv, t, d = 2, 4, 2, 19, 32
    pi = rotation.dense_rotation(1, d)
    smat = rng.round_to_bf16(rng.normals(2, d * d).reshape(d, d))
    kq, vq, kc, vc = _quantized_cache(b, hkv, t, d, 3, pi, smat, 4, 2)
    q = np.random.default_rng(5).standard_normal((b, hq, d))
    start = np.array([18, 6])
    out = attention.prefill(q[:, None], kc, vc, start, pi, smat, kq["centroids"], vq["centroids"])
    want, _ = attention.decode(q, kc, vc, start + 1, pi, smat, kq["centroids"], vq["centroids"])
    assert np.array_equal(out[:, 0], want)
