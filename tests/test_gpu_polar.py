"""GPU parity of the PolarQuant variant (keys as recursive polar angles) against
the fp64 oracle (oracle/polar.py), through the C ABI: the quantize kernel's
angle codes and norms for every code width, both rotations, bf16 and fp32
input, ragged counts, edge vectors (exact zeros in the rotated vector, the
cut at +-pi, zero and saturated norms, fp16 midpoints) and the slot modes;
the decode scan's logits and outputs on the oracle's codes for every
supported width pair, GQA group and ragged lengths; and the GPU's own
quantize followed by decode."""

import numpy as np
import pytest
import torch

import parity_util as P
from oracle import codebook as ocb
from oracle import polar as op
from oracle import quantize as oq
from online_kv_cache_quantize_gb300 import binding as B
from online_kv_cache_quantize_gb300 import workloads as W

pytestmark = pytest.mark.gpu

D = 128
LOGIT_TOL = 1e-4
OUT_TOL = 1e-3
# an fp64 angle this close to a boundary may be decided either way: atan2 and
# hypot of the GPU and of the host differ in the last ulps, and with bf16
# input the RHT rotation cancels exactly now and then, putting a level-1
# angle exactly on a multiple of pi/4 (a boundary at 3 and 4 bits) or on the
# cut at +-pi, where the oracle's rounded matrix product leaves a residue of
# 1e-16 that the GPU's exact butterflies do not
ANGLE_WINDOW = 1e-12
DECODE_BITS = [(4, 2), (3, 2), (2, 2), (4, 3), (3, 3), (4, 4)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from online_kv_cache_quantize_gb300 import build
    build.build()


def _quantize(x, b1, b2, kind, dtype=torch.bfloat16, rot=None):
    if rot is None:
        rot, _ = P.handles(D, kind)
    xt = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda().to(dtype)
    cache = B.Cache("polar", b1, D, rows=1, capacity=max(xt.shape[0], 1), bits2=b2)
    B.tq_quantize_kv(cache, rot, xt)
    torch.cuda.synchronize()
    return cache


def _compare(cache, x64, b1, b2, kind, label, bound_exempt=True):
    """Codes identical to the oracle's (exempt: an fp64 angle within
    ANGLE_WINDOW of a boundary, each listed), packed layout exact, fp16
    norms identical except next to a rounding midpoint."""
    n = x64.shape[0]
    pi, _ = P.oracle_mats(D, kind)
    qz = op.quantize(x64, pi, b1, b2)
    got = cache.codes[:n].cpu().numpy()
    gidx = op.unpack(got, D, b1, b2)
    assert np.array_equal(op.pack(gidx, D, b1, b2), got), f"{label}: packed layout differs"
    mism_total = 0
    for lev, (gi, oi, ang) in enumerate(zip(gidx, qz["idx"], qz["angles"]), start=1):
        _, t = op.codebook(lev, b1 if lev == 1 else b2)
        if lev == 1:  # the cut at +-pi is the edge between the last and the first cell
            t = np.concatenate([t, [-np.pi, np.pi]])
        near = np.any(np.abs(ang[..., None] - t) <= ANGLE_WINDOW, axis=-1) if t.size else np.zeros_like(gi, bool)
        mism = gi != oi
        for r, j in np.argwhere(mism):
            print(f"{label}: exempt angle mismatch level {lev} row {r} angle {j}: psi = {ang[r, j]!r}, "
                  f"codes gpu {gi[r, j]} / oracle {oi[r, j]}")
        bad = mism & ~near
        assert not bad.any(), f"{label}: level {lev}: {bad.sum()} angle codes differ, e.g. {np.argwhere(bad)[:5].tolist()}"
        mism_total += int(mism.sum())
    angles = n * (D - 1)
    if bound_exempt:  # random data: exact ties are rare
        assert mism_total <= 1e-5 * angles + 1, f"{label}: too many exempt angle mismatches ({mism_total})"
    gn = cache.norm[:n].cpu().numpy().view(np.float16).astype(np.float64)
    nbad = (gn != qz["norm16"]) & ~P._near_fp16_midpoint(qz["n"], P.NORM_WINDOW)
    assert not nbad.any(), f"{label}: {nbad.sum()} fp16 norms differ, e.g. rows {np.flatnonzero(nbad)[:5].tolist()}"
    return mism_total


@pytest.mark.parametrize("kind", ["rht", "dense"])
@pytest.mark.parametrize("b1,b2", [(4, 2), (3, 2), (2, 2), (4, 3), (1, 1), (4, 4), (2, 1), (3, 4)])
def test_quantize_every_width(kind, b1, b2):
    """2 KV heads x 1000 tokens of the decode law (outlier channels, LogNormal
    token scale, 1 % heavy tokens), bf16 input."""
    k, _ = W.decode_kv(1, 2, 1000, heavy_frac=0.01, seed=b1 * 10 + b2)
    x = W.round_bf16(k.reshape(-1, D))
    cache = _quantize(x, b1, b2, kind)
    _compare(cache, x.astype(np.float64), b1, b2, kind, f"polar-{kind}-{b1}{b2}")


@pytest.mark.parametrize("kind", ["rht", "dense"])
def test_quantize_fp32_input_ragged(kind):
    """fp32 input, N(0, 1) x LogNormal scale, 1237 vectors (ragged grid tail)."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((1237, D)) * rng.lognormal(0, 1, (1237, 1))).astype(np.float32)
    cache = _quantize(x, 4, 2, kind, dtype=torch.float32)
    _compare(cache, x.astype(np.float64), 4, 2, kind, f"polar-f32-{kind}")


def test_quantize_edge_vectors():
    """Zero vector, one-hot, two equal entries (exact zeros in the RHT-rotated
    vector: pairs on the axes and at the cut), tiny and saturating norms,
    fp16-midpoint norms, among ordinary rows."""
    n = 200
    x = W.round_bf16(np.random.default_rng(8).standard_normal((n, D)).astype(np.float32))
    x[0] = 0.0
    x[1] = 0.0
    x[1, 7] = 1.0
    x[2] = 0.0
    x[2, 0] = x[2, 1] = 3.0
    x[3] = 0.0
    x[3, 0], x[3, 1] = 2.0, -2.0
    x[4] = 0.0
    x[4, 5] = x[4, 9] = x[4, 66] = -1.0
    x[5] = 2.0 ** -100
    x[6] = 8192.0
    x[7] = -1.0
    x[8] = 0.0
    x[8, 5] = 3 * 2.0 ** -25      # norm 3 * 2^-25: an fp16 subnormal midpoint
    x[9] = 0.0
    x[9, 30], x[9, 31] = 65.0, -2112.0   # norm 2113: between 2112 and 2114
    assert np.array_equal(W.round_bf16(x), x)
    for kind in ("rht", "dense"):
        for b1, b2 in ((4, 2), (3, 3), (1, 2)):
            cache = _quantize(x, b1, b2, kind)
            # constant and sparse rows put RHT angles exactly on boundaries by construction
            _compare(cache, x.astype(np.float64), b1, b2, kind, f"polar-edge-{kind}-{b1}{b2}", bound_exempt=False)
            gn = cache.norm[:n].cpu().numpy().view(np.float16).astype(np.float64)
            # planted midpoints: the fp16 of the exact norm, ties to even
            assert gn[0] == 0.0 and gn[6] == 65504.0
            assert gn[8] == oq.fp16_rne(np.float64(3 * 2.0 ** -25)) and gn[9] == oq.fp16_rne(np.float64(2113.0))


def test_quantize_slot_modes_and_strided_rows():
    """dst_slot scatter (skipped slots), append_pos and rows with a stride of
    192 elements give the contiguous call's bytes."""
    n = 640
    rot, _ = P.handles(D, "rht")
    x = W.round_bf16(np.random.default_rng(21).standard_normal((n, D)).astype(np.float32))
    xt = torch.from_numpy(x).cuda().to(torch.bfloat16)
    ref = B.Cache("polar", 4, D, rows=1, capacity=n, bits2=2)
    B.tq_quantize_kv(ref, rot, xt)
    wide = torch.zeros((n, 192), dtype=torch.bfloat16, device="cuda")
    wide[:, 32:32 + D] = xt
    st = B.Cache("polar", 4, D, rows=1, capacity=n, bits2=2)
    B.tq_quantize_kv(st, rot, wide[:, 32:32 + D])
    cap = 3 * n + 1
    dst = (3 * torch.arange(n, dtype=torch.int64, device="cuda")) % cap
    dst[::7] = -1
    sc = B.Cache("polar", 4, D, rows=1, capacity=cap, bits2=2)
    B.tq_quantize_kv(sc, rot, xt, dst_slot=dst)
    heads, cap2 = 4, 24
    pos = torch.from_numpy(np.random.default_rng(2).integers(0, cap2, n // heads).astype(np.int32)).cuda()
    pos[5] = -1
    ac = B.Cache("polar", 4, D, rows=n, capacity=cap2, bits2=2)
    B.tq_quantize_kv(ac, rot, xt, append_pos=pos, heads=heads)
    torch.cuda.synchronize()
    assert torch.equal(st.codes, ref.codes) and torch.equal(st.norm, ref.norm)
    keep = torch.nonzero(dst >= 0).flatten()
    assert torch.equal(sc.codes[dst[keep]], ref.codes[keep]) and torch.equal(sc.norm[dst[keep]], ref.norm[keep])
    untouched = torch.ones(cap, dtype=torch.bool, device="cuda")
    untouched[dst[keep]] = False
    assert int(sc.codes[untouched].abs().sum()) == 0
    v = torch.arange(n, device="cuda")
    pv = pos[v // heads].long()
    ok = pv >= 0
    slots = v[ok] * cap2 + pv[ok]
    assert torch.equal(ac.codes[slots], ref.codes[v[ok]]) and torch.equal(ac.norm[slots], ref.norm[v[ok]])


# ------------------------------------------------------------------ decode --
def _oracle_caches(k, v, b1, b2, vbits, kind):
    """PolarQuant keys and MSE values quantized and packed by the ORACLE,
    uploaded into GPU caches."""
    bsz, hkv, cap, _ = k.shape
    pi, _ = P.oracle_mats(D, kind)
    kq = op.quantize(k.reshape(-1, D).astype(np.float64), pi, b1, b2)
    packed = op.pack(kq["idx"], D, b1, b2)
    vq = oq.quantize(v.reshape(-1, D).astype(np.float64), pi, "mse", vbits)
    gk = B.Cache("polar", b1, D, rows=bsz * hkv, capacity=cap, bits2=b2)
    gk.codes.copy_(torch.from_numpy(packed))
    gk.norm.copy_(torch.from_numpy(kq["norm16"].astype(np.float16).view(np.int16)))
    gv = P.oracle_cache_planes(vq, "mse", vbits, bsz * hkv, cap)
    sh = (bsz, hkv, cap)
    kc = {"packed": packed.reshape(sh + (-1,)), "norm16": kq["norm16"].reshape(sh)}
    vc = {"idx": vq["idx"].reshape(sh + (D,)), "norm16": vq["norm16"].reshape(sh)}
    return kc, vc, gk, gv, pi


def _gpu_decode(q, gk, gv, lens, kind, n_splits=0, gqa_map=None, out_dtype=torch.float32):
    bsz, hq, _ = q.shape
    rot, _ = P.handles(D, kind)
    qt = torch.from_numpy(np.ascontiguousarray(q, dtype=np.float32)).cuda()
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    maxlen = int(max(lens))
    out = torch.full((bsz, hq, D), float("nan"), dtype=out_dtype, device="cuda")
    logits = torch.full((bsz, hq, max(maxlen, 1)), float("nan"), device="cuda")
    kw = dict(n_splits=n_splits, gqa_map=gqa_map, logits=logits)
    ws = B.workspace(B.tq_attn_decode_workspace(qt, gk, gv, lens_t, maxlen, rot, None, out, **kw))
    B.tq_attn_decode(qt, gk, gv, lens_t, maxlen, rot, None, out, ws, **kw)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), logits.cpu().numpy()


def _check(q, kc, vc, lens, pi, b1, b2, vbits, out, logits, gqa_map=None, out_scale=1.0):
    vcent = ocb.lloyd_max(D, vbits)[0]
    want, wl = op.decode(q.astype(np.float64), kc, vc, lens, pi, b1, b2, vcent, gqa_map=gqa_map)
    bsz, hq, _ = q.shape
    hkv = kc["norm16"].shape[1]
    gmap = np.arange(hq) // (hq // hkv) if gqa_map is None else np.asarray(gqa_map)
    for b in range(bsz):
        for h in range(hq):
            L = lens[b]
            if L == 0:
                assert np.all(out[b, h] == 0)
                continue
            nat = np.linalg.norm(q[b, h]) * kc["norm16"][b, gmap[h], :L] / np.sqrt(D)
            lim = LOGIT_TOL * np.maximum(np.abs(wl[b][h]), nat)
            err = np.abs(logits[b, h, :L] - wl[b][h])
            assert np.all(err <= lim), f"logits b{b} h{h}: max err/lim {np.max(err / lim):.3g}"
            e = np.max(np.abs(out[b, h] - want[b, h]))
            assert e <= OUT_TOL * out_scale, f"out b{b} h{h}: max abs err {e:.3g}"


@pytest.mark.parametrize("kind", ["rht", "dense"])
@pytest.mark.parametrize("b1,b2", DECODE_BITS)
def test_decode_every_width_pair(kind, b1, b2):
    """32 q / 8 KV heads over 1000 tokens (ragged 997 visible), MSE 3-bit values."""
    k, v = W.decode_kv(1, 8, 1000, seed=b1 + 7 * b2)
    kc, vc, gk, gv, pi = _oracle_caches(k, v, b1, b2, 3, kind)
    q = W.query_vectors((1, 32, D), dtype="bf16")
    out, logits = _gpu_decode(q, gk, gv, [997], kind)
    scale = np.max(vc["norm16"]) / np.sqrt(D)
    _check(q, kc, vc, [997], pi, b1, b2, 3, out, logits, out_scale=scale)


@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("vbits", [2, 4])
def test_decode_groups_batches_and_empty(group, vbits):
    """Batch 3 with lengths (0, 1, 300) and several splits; group sizes 1..8."""
    hkv, cap = 2, 320
    k, v = W.decode_kv(3, hkv, cap, heavy_frac=0.05, seed=group)
    kc, vc, gk, gv, pi = _oracle_caches(k, v, 4, 2, vbits, "rht")
    q = W.query_vectors((3, hkv * group, D), seed=group)
    lens = [0, 1, 300]
    out, logits = _gpu_decode(q, gk, gv, lens, "rht", n_splits=3)
    scale = np.max(vc["norm16"]) / np.sqrt(D)
    _check(q, kc, vc, lens, pi, 4, 2, vbits, out, logits, out_scale=scale)


def test_decode_split_invariance_gqa_map_and_bf16_out():
    """One split and automatic splits agree; a permuted GQA map is honoured;
    bf16 output within its rounding of the fp32 one."""
    hkv, cap = 4, 2048
    k, v = W.decode_kv(1, hkv, cap, seed=11)
    kc, vc, gk, gv, pi = _oracle_caches(k, v, 4, 2, 3, "dense")
    q = W.query_vectors((1, 16, D), seed=12)
    gmap = np.array([3, 2, 1, 0] * 4, dtype=np.int32)
    o1, l1 = _gpu_decode(q, gk, gv, [2048], "dense", n_splits=1, gqa_map=gmap)
    o2, l2 = _gpu_decode(q, gk, gv, [2048], "dense", n_splits=0, gqa_map=gmap)
    ob, _ = _gpu_decode(q, gk, gv, [2048], "dense", n_splits=0, gqa_map=gmap, out_dtype=torch.bfloat16)
    scale = np.max(vc["norm16"]) / np.sqrt(D)
    _check(q, kc, vc, [2048], pi, 4, 2, 3, o1, l1, gqa_map=gmap, out_scale=scale)
    _check(q, kc, vc, [2048], pi, 4, 2, 3, o2, l2, gqa_map=gmap, out_scale=scale)
    assert np.array_equal(l1, l2)
    assert np.max(np.abs(o1 - o2)) <= 1e-5 * scale
    assert np.max(np.abs(ob - o2)) <= 2.0 ** -8 * np.max(np.abs(o2)) + 1e-6


def test_gpu_quantize_then_decode():
    """1 x 32 q / 8 KV heads x 8192 tokens: the GPU quantizes the PolarQuant
    keys (4 / 2 bits) and the 3-bit MSE values itself, then decodes; sampled
    query heads against the oracle end to end."""
    hkv, L = 8, 8192
    k, v = W.decode_kv(1, hkv, L, seed=5)
    rot, _ = P.handles(D, "rht")
    gk = B.Cache("polar", 4, D, rows=hkv, capacity=L, bits2=2)
    gv = B.Cache("mse", 3, D, rows=hkv, capacity=L)
    B.tq_quantize_kv(gk, rot, torch.from_numpy(k.reshape(-1, D)).cuda().to(torch.bfloat16))
    B.tq_quantize_kv(gv, rot, torch.from_numpy(v.reshape(-1, D)).cuda().to(torch.bfloat16))
    torch.cuda.synchronize()
    # every key code of the fill against the oracle first (the decode check
    # below assumes the two caches hold the same codes)
    _compare(gk, k.reshape(-1, D).astype(np.float64), 4, 2, "rht", "polar-fill-8x8192")
    q = W.query_vectors((1, 32, D), dtype="bf16", seed=6)
    out, logits = _gpu_decode(q, gk, gv, [L], "rht")
    pi, _ = P.oracle_mats(D, "rht")
    vcent = ocb.lloyd_max(D, 3)[0]
    gcodes = gk.codes.cpu().numpy().reshape(hkv, L, -1)
    for h in (0, 9, 31):
        kv = h // 4
        kq = op.quantize(W.round_bf16(k[0, kv]).astype(np.float64), pi, 4, 2)
        vq = oq.quantize(W.round_bf16(v[0, kv]).astype(np.float64), pi, "mse", 3)
        opk = op.pack(kq["idx"], D, 4, 2)
        # tokens whose codes hold an exempt tie (checked and listed by _compare
        # above) have two valid logits: those are left out of the logit check
        same = np.all(opk == gcodes[kv], axis=1)
        kc = {"packed": opk[None, None], "norm16": kq["norm16"][None, None]}
        vc = {"idx": vq["idx"][None, None], "norm16": vq["norm16"][None, None]}
        want, wl = op.decode(q[:, h:h + 1].astype(np.float64), kc, vc, [L], pi, 4, 2, vcent)
        scale = np.max(vq["norm16"]) / np.sqrt(D)
        assert np.max(np.abs(out[0, h] - want[0, 0])) <= OUT_TOL * scale, h
        nat = np.linalg.norm(q[0, h]) * kq["norm16"] / np.sqrt(D)
        err = np.abs(logits[0, h] - wl[0][0]) / (LOGIT_TOL * np.maximum(np.abs(wl[0][0]), nat))
        assert same.sum() >= L - 16
        bad = np.flatnonzero((err > 1) & same)
        assert bad.size == 0, (h, bad[:10].tolist(), err[bad[:10]].tolist(), logits[0, h, bad[:5]].tolist(),
                               wl[0][0][bad[:5]].tolist())


def test_unsupported_calls_are_refused():
    """PolarQuant keys in the step, prefill and search entry points, a decode
    width pair without a scan kernel, and a PolarQuant value cache: each
    returns TQ_ERR_UNSUPPORTED before any launch."""
    hkv, cap = 1, 64
    k, v = W.decode_kv(1, hkv, cap)
    kc, vc, gk, gv, pi = _oracle_caches(k, v, 4, 2, 3, "rht")
    rot, qjl = P.handles(D, "rht")
    q = torch.from_numpy(W.query_vectors((1, 4, D))).cuda()
    lens = torch.tensor([cap], dtype=torch.int32, device="cuda")
    out = torch.empty((1, 4, D), device="cuda")
    ws = B.workspace(1 << 20)
    with pytest.raises(B.TQError) as e:
        B.tq_decode_step(q, gk, gv, lens, cap, rot, qjl, out, q[0, :1].contiguous(), q[0, :1].contiguous(),
                         torch.zeros(1, dtype=torch.int32, device="cuda"), ws)
    assert "UNSUPPORTED" in str(e.value)
    odd = B.Cache("polar", 1, D, rows=hkv, capacity=cap, bits2=1)
    with pytest.raises(B.TQError) as e:
        B.tq_attn_decode(q, odd, gv, lens, cap, rot, None, out, ws)
    assert "UNSUPPORTED" in str(e.value)
    with pytest.raises(B.TQError) as e:
        B.tq_attn_decode(q, gk, gk, lens, cap, rot, None, out, ws)
    assert "UNSUPPORTED" in str(e.value)
    qp = torch.from_numpy(W.query_vectors((1, 2, 4, D))).cuda()
    op_ = torch.empty((1, 2, 4, D), device="cuda")
    qs = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(B.TQError) as e:
        B.tq_attn_prefill(qp, gk, gv, qs, cap, rot, qjl, op_, ws)
    assert "UNSUPPORTED" in str(e.value)


def test_alternating_polar_and_turboquant_decodes_on_one_thread():
    """The library reuses the last prepared decode call of a thread when the
    arguments repeat: alternating PolarQuant and TurboQuant key caches (and
    repeating each) must give each call its own kernels and the same outputs
    as the first run."""
    hkv, cap = 2, 256
    k, v = W.decode_kv(1, hkv, cap, seed=31)
    kc, vc, gk, gv, pi = _oracle_caches(k, v, 4, 2, 3, "rht")
    rot, qjl = P.handles(D, "rht")
    tk = B.Cache("prod", 3, D, rows=hkv, capacity=cap)
    B.tq_quantize_kv(tk, rot, torch.from_numpy(k.reshape(-1, D)).cuda().to(torch.bfloat16), qjl=qjl)
    q = torch.from_numpy(W.query_vectors((1, 8, D), seed=32)).cuda()
    lens = torch.tensor([200], dtype=torch.int32, device="cuda")
    outs = {}
    for rep in range(3):
        for name, kcache, qj in (("polar", gk, None), ("turbo", tk, qjl)):
            out = torch.empty((1, 8, D), device="cuda")
            ws = B.workspace(B.tq_attn_decode_workspace(q, kcache, gv, lens, cap, rot, qj, out))
            B.tq_attn_decode(q, kcache, gv, lens, cap, rot, qj, out, ws)
            B.tq_attn_decode(q, kcache, gv, lens, cap, rot, qj, out, ws)  # the same arguments again
            torch.cuda.synchronize()
            if rep == 0:
                outs[name] = out.clone()
            else:
                assert torch.equal(out, outs[name]), (name, rep)
    assert not torch.equal(outs["polar"], outs["turbo"])
