"""GPU parity of decode attention (logits and outputs) against the fp64 oracle.

The caches the GPU decodes here are packed by the ORACLE and uploaded, so
the decode half is checked on exactly the oracle's codes. A separate test
runs the GPU's own quantize followed by decode at the full decode shape.
"""

import numpy as np
import pytest
import torch

import parity_util as P
from oracle import attention as oa
from oracle import quantize as oq
from online_kv_cache_quantize_gb300 import binding as B
from online_kv_cache_quantize_gb300 import workloads as W

pytestmark = pytest.mark.gpu

LOGIT_TOL = 1e-4
OUT_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from online_kv_cache_quantize_gb300 import build
    build.build()


def _oracle_caches(k, v, kbits, vbits, kind, d=128, kbits2=None, vbits2=None):
    """Oracle-quantized caches: returns (unpacked dicts, GPU caches, oracle qz);
    kbits2 / vbits2: the second channel group's bits of fractional-rate caches."""
    bsz, hkv, cap, _ = k.shape
    pi, s = P.oracle_mats(d, kind)
    kq = oq.quantize(k.reshape(-1, d).astype(np.float64), pi, "prod", kbits, s, bits2=kbits2)
    vq = oq.quantize(v.reshape(-1, d).astype(np.float64), pi, "mse", vbits, bits2=vbits2)
    sh = (bsz, hkv, cap)
    kc = {"idx": kq["idx"].reshape(sh + (d,)), "norm16": kq["norm16"].reshape(sh),
          "rnorm16": kq["rnorm16"].reshape(sh), "z": kq["z"].reshape(sh + (d,))}
    vc = {"idx": vq["idx"].reshape(sh + (d,)), "norm16": vq["norm16"].reshape(sh)}
    gk = P.oracle_cache_planes(kq, "prod", kbits, bsz * hkv, cap, bits2=kbits2)
    gv = P.oracle_cache_planes(vq, "mse", vbits, bsz * hkv, cap, bits2=vbits2)
    return kc, vc, gk, gv, kq, vq, pi, s


def _gpu_decode(q, gk, gv, lens, kind, n_splits=0, gqa_map=None, out_dtype=torch.float32, with_logits=True):
    bsz, hq, d = q.shape
    rot, qjl = P.handles(d, kind)
    qt = torch.from_numpy(np.ascontiguousarray(q, dtype=np.float32)).cuda()
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    maxlen = int(max(lens)) if len(lens) else 0
    out = torch.full((bsz, hq, d), float("nan"), dtype=out_dtype, device="cuda")
    logits = torch.full((bsz, hq, max(maxlen, 1)), float("nan"), device="cuda") if with_logits else None
    kw = dict(n_splits=n_splits, gqa_map=gqa_map, logits=logits)
    ws = B.workspace(B.tq_attn_decode_workspace(qt, gk, gv, lens_t, maxlen, rot, qjl, out, **kw))
    B.tq_attn_decode(qt, gk, gv, lens_t, maxlen, rot, qjl, out, ws, **kw)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), (logits.cpu().numpy() if with_logits else None)


def _check(q, kc, vc, kq, vq, lens, pi, s, out, logits, gqa_map=None, out_scale=1.0):
    want, want_logits = oa.decode(q.astype(np.float64), kc, vc, lens, pi, s, kq["centroids"], vq["centroids"],
                                  gqa_map=gqa_map)
    bsz, hq, d = q.shape
    hkv = kc["idx"].shape[1]
    gmap = oa.default_gqa_map(hq, hkv) if gqa_map is None else np.asarray(gqa_map)
    for b in range(bsz):
        for h in range(hq):
            L = lens[b]
            if L == 0:
                assert np.all(out[b, h] == 0)
                continue
            if logits is not None:
                kv = gmap[h]
                nat = np.linalg.norm(q[b, h]) * kc["norm16"][b, kv, :L] / np.sqrt(d)
                lim = LOGIT_TOL * np.maximum(np.abs(want_logits[b][h]), nat)
                err = np.abs(logits[b, h, :L] - want_logits[b][h])
                assert np.all(err <= lim), f"logits b{b} h{h}: max err/lim {np.max(err / lim):.3g}"
            e = np.max(np.abs(out[b, h] - want[b, h]))
            assert e <= OUT_TOL * out_scale, f"out b{b} h{h}: max abs err {e:.3g} > {OUT_TOL * out_scale:.3g}"


def test_single_head_logits_dense():
    """Outlier keys (4096 x 128, x20 channels), 3-bit PROD, dense QR, logits of one query."""
    x, _ = W.outlier_keys(4096, 128)
    k = x.reshape(1, 1, 4096, 128)
    v = np.random.default_rng(5).standard_normal((1, 1, 4096, 128)).astype(np.float32)
    kc, vc, gk, gv, kq, vq, pi, s = _oracle_caches(k, v, 3, 3, "dense")
    q = W.query_vectors((1, 1, 128))
    out, logits = _gpu_decode(q, gk, gv, [4096], "dense")
    _check(q, kc, vc, kq, vq, [4096], pi, s, out, logits)


@pytest.mark.parametrize("kbits,vbits", [(3, 3), (4, 4), (2, 2), (3, 4), (5, 1)])
@pytest.mark.parametrize("kind", ["rht", "dense"])
def test_gqa4_unit_scale(kbits, vbits, kind):
    """32 q / 8 KV heads, unit-scale N(0,1) data, ragged length."""
    r = np.random.default_rng(kbits * 10 + vbits)
    k = W.round_bf16(r.standard_normal((1, 8, 1008, 128)).astype(np.float32))
    v = W.round_bf16(r.standard_normal((1, 8, 1008, 128)).astype(np.float32))
    kc, vc, gk, gv, kq, vq, pi, s = _oracle_caches(k, v, kbits, vbits, kind)
    q = W.query_vectors((1, 32, 128), dtype="bf16")
    out, logits = _gpu_decode(q, gk, gv, [997], kind)
    _check(q, kc, vc, kq, vq, [997], pi, s, out, logits)


@pytest.mark.parametrize("group", [1, 2, 8])
def test_group_sizes_batch_and_empty(group):
    """Batch 3 with lengths (0, 1, 300); group sizes 1, 2, 8; outlier data."""
    hkv, cap = 2, 320
    k, v = W.decode_kv(3, hkv, cap, heavy_frac=0.05)
    kc, vc, gk, gv, kq, vq, pi, s = _oracle_caches(k, v, 3, 4, "rht")
    q = W.query_vectors((3, hkv * group, 128))
    lens = [0, 1, 300]
    out, logits = _gpu_decode(q, gk, gv, lens, "rht")
    scale = np.max(vc["norm16"]) / np.sqrt(128)
    _check(q, kc, vc, kq, vq, lens, pi, s, out, logits, out_scale=scale)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_many_rows_few_splits(out_dtype):
    """Batch 8 x 32 query heads (256 rows) over 512 tokens: few splits per
    row, so the warp-per-row merge runs; RHT and dense."""
    for kind in ("rht", "dense"):
        k, v = W.decode_kv(8, 4, 512, seed=41)
        kc, vc, gk, gv, kq, vq, pi, s = _oracle_caches(k, v, 3, 3, kind)
        q = W.query_vectors((8, 32, 128), seed=42)
        lens = [512, 1, 0, 300, 511, 64, 65, 200]
        out, logits = _gpu_decode(q, gk, gv, lens, kind, out_dtype=out_dtype, with_logits=out_dtype == torch.float32)
        scale = np.max(vc["norm16"]) / np.sqrt(128)
        if out_dtype == torch.float32:
            _check(q, kc, vc, kq, vq, lens, pi, s, out, logits, out_scale=scale)
        else:
            want, _ = oa.decode(q.astype(np.float64), kc, vc, lens, pi, s, kq["centroids"], vq["centroids"])
            assert np.max(np.abs(out - want)) <= 2.0**-8 * np.max(np.abs(want)) + OUT_TOL * scale


def test_split_invariance_and_gqa_map():
    """n_splits = 1 and automatic splits agree; a permuted GQA map is honoured."""
    hkv, cap = 4, 2048
    k, v = W.decode_kv(1, hkv, cap)
    kc, vc, gk, gv, kq, vq, pi, s = _oracle_caches(k, v, 4, 4, "dense")
    q = W.query_vectors((1, 16, 128))
    gmap = np.array([3, 2, 1, 0] * 4, dtype=np.int32)
    o1, l1 = _gpu_decode(q, gk, gv, [2048], "dense", n_splits=1, gqa_map=gmap)
    o2, l2 = _gpu_decode(q, gk, gv, [2048], "dense", n_splits=0, gqa_map=gmap)
    o3, _ = _gpu_decode(q, gk, gv, [2048], "dense", n_splits=37, gqa_map=gmap, with_logits=False)
    scale = np.max(vc["norm16"]) / np.sqrt(128)
    _check(q, kc, vc, kq, vq, [2048], pi, s, o1, l1, gqa_map=gmap, out_scale=scale)
    _check(q, kc, vc, kq, vq, [2048], pi, s, o2, l2, gqa_map=gmap, out_scale=scale)
    assert np.max(np.abs(o1 - o2)) <= 1e-5 * scale and np.max(np.abs(o1 - o3)) <= 1e-5 * scale
    assert np.array_equal(l1, l2)


def test_capacity_must_be_multiple_of_16():
    k, v = W.decode_kv(1, 1, 40)
    kc, vc, gk, gv, kq, vq, pi, s = _oracle_caches(k, v, 3, 3, "rht")
    with pytest.raises(B.TQError) as e:
        _gpu_decode(W.query_vectors((1, 1, 128)), gk, gv, [40], "rht")
    assert "ALIGNMENT" in str(e.value)


def test_bf16_output():
    k, v = W.decode_kv(1, 2, 256)
    kc, vc, gk, gv, kq, vq, pi, s = _oracle_caches(k, v, 3, 3, "rht")
    q = W.query_vectors((1, 8, 128))
    out, _ = _gpu_decode(q, gk, gv, [256], "rht", out_dtype=torch.bfloat16, with_logits=False)
    want, _ = oa.decode(q.astype(np.float64), kc, vc, [256], pi, s, kq["centroids"], vq["centroids"])
    assert np.max(np.abs(out - want)) <= 2.0**-8 * np.max(np.abs(want)) + OUT_TOL


def test_full_decode_shape_gpu_quantize_then_decode():
    """Decode shape of a Llama-3.1-8B step (1 x 32 q / 8 KV heads x 32768 tokens),
    the GPU quantizing the cache itself (RHT, K 3-bit PROD / V 3-bit MSE),
    sampled query heads checked against the oracle end to end."""
    d, hkv, L = 128, 8, 32768
    k, v = W.decode_kv(1, hkv, L)
    rot, qjl = P.handles(d, "rht")
    gk = B.Cache("prod", 3, d, rows=hkv, capacity=L)
    gv = B.Cache("mse", 3, d, rows=hkv, capacity=L)
    B.tq_quantize_kv(gk, rot, torch.from_numpy(k.reshape(-1, d)).cuda().to(torch.bfloat16), qjl=qjl)
    B.tq_quantize_kv(gv, rot, torch.from_numpy(v.reshape(-1, d)).cuda().to(torch.bfloat16))
    q = W.query_vectors((1, 32, d), dtype="bf16")
    out, _ = _gpu_decode(q, gk, gv, [L], "rht", with_logits=False)
    pi, s = P.oracle_mats(d, "rht")
    scale = None
    for h in (0, 13, 31):
        kv = h // 4
        kq = oq.quantize(k[0, kv].astype(np.float64), pi, "prod", 3, s)
        vq = oq.quantize(v[0, kv].astype(np.float64), pi, "mse", 3)
        qp, u = oa.query_prep(q[0, h].astype(np.float64), pi, s)
        l = oa.key_logits(qp, u, kq["idx"], kq["norm16"], kq["centroids"], kq["rnorm16"], kq["z"], d)
        vhat = vq["norm16"][:, None] * vq["centroids"][vq["idx"]]
        sc = l / np.sqrt(d)
        p = np.exp(sc - sc.max())
        p /= p.sum()
        want = (p @ vhat) @ pi
        scale = np.max(vq["norm16"]) / np.sqrt(d)
        assert np.max(np.abs(out[0, h] - want)) <= OUT_TOL * scale, h


@pytest.mark.parametrize("kbits,vbits", [(3, 3), (4, 4), (5, 4), (3, 2), (4, 2)])
@pytest.mark.parametrize("kind", ["rht", "dense"])
def test_fractional_rate_caches(kbits, vbits, kind):
    """Two-group caches (coordinates with i % 16 < 8 at bits, the rest at
    bits - 1): keys PROD 3/2 and values MSE 3/2 make the 2.5-bit cache, 4/3 and
    4/3 the 3.5-bit one; 32 q / 8 KV heads, outlier data, ragged length."""
    k, v = W.decode_kv(1, 8, 1008, heavy_frac=0.05, seed=kbits * 10 + vbits)
    kc, vc, gk, gv, kq, vq, pi, s = _oracle_caches(k, v, kbits, vbits, kind, kbits2=kbits - 1, vbits2=vbits - 1)
    q = W.query_vectors((1, 32, 128), dtype="bf16")
    out, logits = _gpu_decode(q, gk, gv, [997], kind)
    scale = np.max(vc["norm16"]) / np.sqrt(128)
    _check(q, kc, vc, kq, vq, [997], pi, s, out, logits, out_scale=scale)


@pytest.mark.parametrize("group", [1, 8])
def test_fractional_rate_group_sizes_and_batch(group):
    """2.5-bit caches, batch 3 with lengths (0, 17, 300), group sizes 1 and 8."""
    hkv, cap = 2, 320
    k, v = W.decode_kv(3, hkv, cap, heavy_frac=0.05)
    kc, vc, gk, gv, kq, vq, pi, s = _oracle_caches(k, v, 3, 3, "rht", kbits2=2, vbits2=2)
    q = W.query_vectors((3, hkv * group, 128))
    lens = [0, 17, 300]
    out, logits = _gpu_decode(q, gk, gv, lens, "rht")
    scale = np.max(vc["norm16"]) / np.sqrt(128)
    _check(q, kc, vc, kq, vq, lens, pi, s, out, logits, out_scale=scale)


def test_fractional_rate_mixed_caches_rejected():
    """Keys at a fractional rate with whole-width values (or the reverse) are
    not taken: TQ_ERR_UNSUPPORTED, nothing launched."""
    k, v = W.decode_kv(1, 2, 64)
    for kb2, vb2 in ((2, None), (None, 2)):
        kc, vc, gk, gv, kq, vq, pi, s = _oracle_caches(k, v, 3, 3, "rht", kbits2=kb2, vbits2=vb2)
        with pytest.raises(B.TQError) as e:
            _gpu_decode(W.query_vectors((1, 8, 128)), gk, gv, [64], "rht")
        assert "UNSUPPORTED" in str(e.value)
