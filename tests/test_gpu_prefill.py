"""GPU parity of chunked-prefill attention against the fp64 oracle.

The caches are packed by the ORACLE and uploaded (as in the decode tests), so
the prefill kernel is checked on exactly the oracle's codes; one test at the
Llama-3.1-8B prefill shape lets the GPU quantize the cache itself and checks
sampled query rows.
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

OUT_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from online_kv_cache_quantize_gb300 import build
    build.build()


def _caches(k, v, kbits, vbits, kind, kbits2=None, vbits2=None):
    d = k.shape[-1]
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


def _gpu_prefill(q, gk, gv, q_start, max_context, kind, n_splits=0, out_dtype=torch.float32, q_dtype=torch.float32,
                 gqa_map=None):
    bsz, c, hq, d = q.shape
    rot, qjl = P.handles(d, kind)
    qt = torch.from_numpy(np.ascontiguousarray(q, dtype=np.float32)).cuda().to(q_dtype)
    qs = torch.tensor(q_start, dtype=torch.int32, device="cuda")
    out = torch.full((bsz, c, hq, d), float("nan"), dtype=out_dtype, device="cuda")
    kw = dict(n_splits=n_splits, gqa_map=gqa_map)
    ws = B.workspace(B.tq_attn_prefill_workspace(qt, gk, gv, qs, max_context, rot, qjl, out, **kw))
    B.tq_attn_prefill(qt, gk, gv, qs, max_context, rot, qjl, out, ws, **kw)
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def _check(q, kc, vc, kq, vq, q_start, pi, s, out, gqa_map=None):
    want = oa.prefill(q.astype(np.float64), kc, vc, q_start, pi, s, kq["centroids"], vq["centroids"], gqa_map=gqa_map)
    scale = max(np.max(vc["norm16"]) / np.sqrt(q.shape[-1]), 1e-30)
    err = np.max(np.abs(out - want))
    assert err <= OUT_TOL * scale, f"max abs err {err:.3g} > {OUT_TOL * scale:.3g}"
    return want


@pytest.mark.parametrize("kbits,vbits", [(3, 3), (4, 4), (2, 2), (5, 1)])
@pytest.mark.parametrize("kind", ["rht", "dense"])
def test_prefill_gqa4_ragged(kbits, vbits, kind):
    """Batch 2, 8 q / 2 KV heads, chunk of 40 tokens (160 rows per KV head: two
    full CTAs of 64 rows and a ragged third), one chunk ending at the capacity
    and one mid-cache; outlier data."""
    k, v = W.decode_kv(2, 2, 1024, heavy_frac=0.05, seed=kbits * 10 + vbits)
    kc, vc, gk, gv, kq, vq, pi, s = _caches(k, v, kbits, vbits, kind)
    q = W.query_vectors((2, 40, 8, 128), dtype="bf16", seed=7)
    q_start = [984, 300]
    out = _gpu_prefill(q, gk, gv, q_start, 1024, kind)
    _check(q, kc, vc, kq, vq, q_start, pi, s, out)


@pytest.mark.parametrize("group,chunk", [(1, 17), (2, 33), (8, 9)])
def test_prefill_group_sizes(group, chunk):
    """Query heads per KV head 1, 2, 8 with chunks that leave ragged CTAs."""
    hkv, cap = 2, 512
    k, v = W.decode_kv(1, hkv, cap, seed=group)
    kc, vc, gk, gv, kq, vq, pi, s = _caches(k, v, 3, 4, "rht")
    q = W.query_vectors((1, chunk, hkv * group, 128), seed=8)
    q_start = [400]
    out = _gpu_prefill(q, gk, gv, q_start, cap, "rht")
    _check(q, kc, vc, kq, vq, q_start, pi, s, out)


def test_prefill_permuted_gqa_map():
    """A permuted query-head -> KV-head map (as decode takes) is honoured."""
    k, v = W.decode_kv(1, 4, 384, seed=31)
    kc, vc, gk, gv, kq, vq, pi, s = _caches(k, v, 3, 3, "dense")
    q = W.query_vectors((1, 20, 16, 128), seed=32)
    gmap = np.array([3, 2, 1, 0] * 4, dtype=np.int32)
    out = _gpu_prefill(q, gk, gv, [364], 384, "dense", gqa_map=gmap)
    _check(q, kc, vc, kq, vq, [364], pi, s, out, gqa_map=gmap)


def test_prefill_first_chunk_causal_triangle():
    """A chunk of 96 tokens at position 0: query i sees only slots 0..i (the
    whole chunk is the causal triangle)."""
    k, v = W.decode_kv(1, 2, 256, seed=3)
    kc, vc, gk, gv, kq, vq, pi, s = _caches(k, v, 3, 3, "rht")
    q = W.query_vectors((1, 96, 8, 128), seed=9)
    out = _gpu_prefill(q, gk, gv, [0], 96, "rht")
    _check(q, kc, vc, kq, vq, [0], pi, s, out)


@pytest.mark.parametrize("kbits,vbits", [(3, 3), (4, 4)])
def test_prefill_fractional_rate_caches(kbits, vbits):
    """2.5-bit (3/2) and 3.5-bit (4/3) caches."""
    k, v = W.decode_kv(1, 2, 640, heavy_frac=0.05, seed=kbits)
    kc, vc, gk, gv, kq, vq, pi, s = _caches(k, v, kbits, vbits, "rht", kbits2=kbits - 1, vbits2=vbits - 1)
    q = W.query_vectors((1, 24, 8, 128), seed=10)
    out = _gpu_prefill(q, gk, gv, [600], 640, "rht")
    _check(q, kc, vc, kq, vq, [600], pi, s, out)


def test_prefill_split_invariance_and_one_token_is_decode():
    """n_splits = 1, automatic and 7 agree; a one-token chunk equals the
    decode kernel's output for the same query and length."""
    hkv, cap = 2, 2048
    k, v = W.decode_kv(1, hkv, cap, seed=11)
    kc, vc, gk, gv, kq, vq, pi, s = _caches(k, v, 3, 3, "dense")
    q = W.query_vectors((1, 8, 8, 128), seed=12)
    o1 = _gpu_prefill(q, gk, gv, [2040], cap, "dense", n_splits=1)
    o2 = _gpu_prefill(q, gk, gv, [2040], cap, "dense")
    o3 = _gpu_prefill(q, gk, gv, [2040], cap, "dense", n_splits=7)
    scale = np.max(vc["norm16"]) / np.sqrt(128)
    assert np.max(np.abs(o1 - o2)) <= 1e-5 * scale and np.max(np.abs(o1 - o3)) <= 1e-5 * scale
    _check(q, kc, vc, kq, vq, [2040], pi, s, o2)
    # one token at position 1500 against decode with length 1501
    q1 = q[:, :1]
    op = _gpu_prefill(q1, gk, gv, [1500], cap, "dense")
    rot, qjl = P.handles(128, "dense")
    qt = torch.from_numpy(np.ascontiguousarray(q1[:, 0], dtype=np.float32)).cuda()
    lens = torch.tensor([1501], dtype=torch.int32, device="cuda")
    od = torch.empty((1, 8, 128), device="cuda")
    ws = B.workspace(B.tq_attn_decode_workspace(qt, gk, gv, lens, cap, rot, qjl, od))
    B.tq_attn_decode(qt, gk, gv, lens, cap, rot, qjl, od, ws)
    torch.cuda.synchronize()
    od = od.cpu().numpy()
    # both against the oracle's decode of length 1501 at the decode output
    # tolerance, and against each other well inside it: the two kernels sum
    # in different orders with different fp16 splits (about 1e-5 of an
    # output of 35 = 1.8 x scale apart)
    want, _ = oa.decode(q1[:, 0].astype(np.float64), kc, vc, [1501], pi, s, kq["centroids"], vq["centroids"])
    assert np.max(np.abs(op[:, 0] - want)) <= OUT_TOL * scale and np.max(np.abs(od - want)) <= OUT_TOL * scale
    assert np.max(np.abs(op[:, 0] - od)) <= 1e-4 * scale


def test_prefill_bf16_io_and_empty_chunk():
    k, v = W.decode_kv(1, 2, 256, seed=13)
    kc, vc, gk, gv, kq, vq, pi, s = _caches(k, v, 3, 3, "rht")
    q = W.query_vectors((1, 16, 8, 128), dtype="bf16", seed=14)
    out = _gpu_prefill(q, gk, gv, [200], 256, "rht", out_dtype=torch.bfloat16, q_dtype=torch.bfloat16)
    want = oa.prefill(q.astype(np.float64), kc, vc, [200], pi, s, kq["centroids"], vq["centroids"])
    assert np.max(np.abs(out - want)) <= 2.0**-8 * np.max(np.abs(want)) + OUT_TOL
    empty = _gpu_prefill(q[:, :0], gk, gv, [200], 256, "rht")
    assert empty.shape == (1, 0, 8, 128)


def test_prefill_rejects_bad_arguments():
    k, v = W.decode_kv(1, 2, 64, seed=15)
    kc, vc, gk, gv, kq, vq, pi, s = _caches(k, v, 3, 3, "rht")
    q = W.query_vectors((1, 4, 8, 128), seed=16)
    with pytest.raises(B.TQError) as e:  # max_context beyond the capacity
        _gpu_prefill(q, gk, gv, [0], 80, "rht")
    assert "CAPACITY" in str(e.value)
    kc2, vc2, gk2, gv2, *_ = _caches(k, v, 3, 3, "rht", kbits2=2)
    with pytest.raises(B.TQError) as e:  # fractional keys with whole-width values
        _gpu_prefill(q, gk2, gv2, [0], 64, "rht")
    assert "UNSUPPORTED" in str(e.value)


def test_prefill_llama8b_chunk_end_of_32k_sampled():
    """Llama-3.1-8B prefill shape: a 512-token chunk at the end of a 32768-token
    context (1 x 32 q / 8 KV heads), the GPU quantizing the cache itself (RHT,
    K 3-bit PROD / V 3-bit MSE); sampled (token, head) rows against the oracle."""
    d, hkv, hq, L, C = 128, 8, 32, 32768, 512
    k, v = W.decode_kv(1, hkv, L)
    rot, qjl = P.handles(d, "rht")
    gk = B.Cache("prod", 3, d, rows=hkv, capacity=L)
    gv = B.Cache("mse", 3, d, rows=hkv, capacity=L)
    B.tq_quantize_kv(gk, rot, torch.from_numpy(k.reshape(-1, d)).cuda().to(torch.bfloat16), qjl=qjl)
    B.tq_quantize_kv(gv, rot, torch.from_numpy(v.reshape(-1, d)).cuda().to(torch.bfloat16))
    q = W.query_vectors((1, C, hq, d), dtype="bf16", seed=17)
    out = _gpu_prefill(q, gk, gv, [L - C], L, "rht", q_dtype=torch.bfloat16)
    pi, s = P.oracle_mats(d, "rht")
    for kv in (0, 5):
        kq = oq.quantize(k[0, kv].astype(np.float64), pi, "prod", 3, s)
        vq = oq.quantize(v[0, kv].astype(np.float64), pi, "mse", 3)
        scale = np.max(vq["norm16"]) / np.sqrt(d)
        for i, j in ((0, 0), (255, 3), (511, 1)):
            h = kv * 4 + j
            n = L - C + i + 1
            qp, u = oa.query_prep(q[0, i, h].astype(np.float64), pi, s)
            l = oa.key_logits(qp, u, kq["idx"][:n], kq["norm16"][:n], kq["centroids"], kq["rnorm16"][:n],
                              kq["z"][:n], d)
            sc = l / np.sqrt(d)
            p = np.exp(sc - sc.max())
            p /= p.sum()
            want = (p @ (vq["norm16"][:n, None] * vq["centroids"][vq["idx"][:n]])) @ pi
            assert np.max(np.abs(out[0, i, h] - want)) <= OUT_TOL * scale, (kv, i, j)


def test_quantized_kv_cache_prefill_chunk_then_step():
    """QuantizedKVCache: prefill 200 / 150 tokens, append a 48-token chunk and
    attend with its queries (against the oracle's causal prefill of the
    combined context), then one decode step continues from the new lengths."""
    d, bsz, hkv, hq, cap, C = 128, 2, 2, 8, 256, 48
    cache = B.QuantizedKVCache(bsz, hq, hkv, cap, k_bits=3, v_bits=3, rotation="rht", rot_seed=W.ROT_SEED,
                               qjl_seed=W.QJL_SEED)
    k, v = W.decode_kv(bsz, hkv, cap, seed=21)
    lens = [200, 150]
    cache.prefill(torch.from_numpy(k[:, :, :200]).cuda(), torch.from_numpy(v[:, :, :200]).cuda(), lens)
    # the chunk's keys and values go to slots lens[b] .. lens[b] + C - 1 of each row
    kc_np = np.stack([k[b, :, lens[b]:lens[b] + C] for b in range(bsz)])
    vc_np = np.stack([v[b, :, lens[b]:lens[b] + C] for b in range(bsz)])
    q = W.query_vectors((bsz, C, hq, d), seed=22)
    out = cache.prefill_chunk(torch.from_numpy(q).cuda(), torch.from_numpy(kc_np).cuda(),
                              torch.from_numpy(vc_np).cuda())
    torch.cuda.synchronize()
    pi, s = P.oracle_mats(d, "rht")
    # the oracle's cache: every row's first lens[b] + C tokens are the ones written
    kq = oq.quantize(k.reshape(-1, d).astype(np.float64), pi, "prod", 3, s)
    vq = oq.quantize(v.reshape(-1, d).astype(np.float64), pi, "mse", 3)
    sh = (bsz, hkv, cap)
    kcd = {"idx": kq["idx"].reshape(sh + (d,)), "norm16": kq["norm16"].reshape(sh),
           "rnorm16": kq["rnorm16"].reshape(sh), "z": kq["z"].reshape(sh + (d,))}
    vcd = {"idx": vq["idx"].reshape(sh + (d,)), "norm16": vq["norm16"].reshape(sh)}
    want = oa.prefill(q.astype(np.float64), kcd, vcd, lens, pi, s, kq["centroids"], vq["centroids"])
    scale = np.max(vq["norm16"]) / np.sqrt(d)
    assert np.max(np.abs(out.cpu().numpy() - want)) <= OUT_TOL * scale
    assert cache.lengths.cpu().tolist() == [lens[0] + C, lens[1] + C]
    # one decode step at the new lengths equals tq_attn_decode over the same cache
    kn = torch.from_numpy(W.round_bf16(W.query_vectors((bsz, hkv, d), seed=23))).cuda()
    vn = torch.from_numpy(W.round_bf16(W.query_vectors((bsz, hkv, d), seed=24))).cuda()
    qd = torch.from_numpy(W.query_vectors((bsz, hq, d), seed=25)).cuda()
    o1 = cache.step(qd, kn, vn).clone()
    new_lens = torch.tensor([lens[0] + C + 1, lens[1] + C + 1], dtype=torch.int32, device="cuda")
    o2 = torch.empty_like(o1)
    ws = B.workspace(B.tq_attn_decode_workspace(qd, cache.k, cache.v, new_lens, cap, cache.rot, cache.qjl, o2))
    B.tq_attn_decode(qd, cache.k, cache.v, new_lens, cap, cache.rot, cache.qjl, o2, ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
