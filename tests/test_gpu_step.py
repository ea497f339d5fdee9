"""tq_decode_step: append the new token's K and V, then decode, in one call.

Checked two ways: bit for bit against the three separate calls on one stream
(tq_quantize_kv K, tq_quantize_kv V, tq_attn_decode), and against the fp64
oracle on the appended cache."""

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


def _setup(bsz, hkv, hq, cap, kind, kbits, vbits, seed, kbits2=0, vbits2=0):
    d = 128
    k, v = W.decode_kv(bsz, hkv, cap, seed=seed)
    rot, qjl = P.handles(d, kind)
    caches = []
    for _ in range(2):
        kc = B.Cache("prod", kbits, d, rows=bsz * hkv, capacity=cap, bits2=kbits2)
        vc = B.Cache("mse", vbits, d, rows=bsz * hkv, capacity=cap, bits2=vbits2)
        B.tq_quantize_kv(kc, rot, torch.from_numpy(k.reshape(-1, d)).cuda().to(torch.bfloat16), qjl=qjl)
        B.tq_quantize_kv(vc, rot, torch.from_numpy(v.reshape(-1, d)).cuda().to(torch.bfloat16))
        caches.append((kc, vc))
    q = torch.from_numpy(W.query_vectors((bsz, hq, d), seed=seed + 1)).cuda()
    knew = torch.from_numpy(W.round_bf16(W.query_vectors((bsz * hkv, d), seed=seed + 2) * 2)).cuda().to(torch.bfloat16)
    vnew = torch.from_numpy(W.round_bf16(W.query_vectors((bsz * hkv, d), seed=seed + 3))).cuda().to(torch.bfloat16)
    return k, v, rot, qjl, caches, q, knew, vnew


@pytest.mark.parametrize("kind,kbits,vbits,frac", [("rht", 3, 3, False), ("dense", 4, 4, False), ("rht", 2, 2, False),
                                                    ("rht", 3, 3, True), ("dense", 4, 4, True)])
def test_step_equals_separate_calls(kind, kbits, vbits, frac):
    """frac: fractional-rate caches (second channel group at bits - 1)."""
    bsz, hkv, hq, cap = 3, 2, 8, 1008
    b2 = dict(kbits2=kbits - 1, vbits2=vbits - 1) if frac else {}
    k, v, rot, qjl, caches, q, knew, vnew = _setup(bsz, hkv, hq, cap, kind, kbits, vbits, seed=40 + kbits, **b2)
    pos = torch.tensor([500, 1007, -1], dtype=torch.int32, device="cuda")  # the third batch row is not appended
    lens = torch.tensor([501, 1008, 700], dtype=torch.int32, device="cuda")
    outs = []
    # separate calls
    (kc, vc) = caches[0]
    B.tq_quantize_kv(kc, rot, knew, qjl=qjl, append_pos=pos, heads=hkv)
    B.tq_quantize_kv(vc, rot, vnew, append_pos=pos, heads=hkv)
    out0 = torch.empty((bsz, hq, 128), device="cuda")
    ws0 = B.workspace(B.tq_attn_decode_workspace(q, kc, vc, lens, cap, rot, qjl, out0))
    B.tq_attn_decode(q, kc, vc, lens, cap, rot, qjl, out0, ws0)
    # one step call
    (kc1, vc1) = caches[1]
    out1 = torch.empty((bsz, hq, 128), device="cuda")
    ws1 = B.workspace(B.tq_decode_step_workspace(q, kc1, vc1, lens, cap, rot, qjl, out1, knew, vnew, pos))
    B.tq_decode_step(q, kc1, vc1, lens, cap, rot, qjl, out1, knew, vnew, pos, ws1)
    torch.cuda.synchronize()
    for name in ("codes", "signs", "norm", "rnorm"):
        assert torch.equal(getattr(kc, name), getattr(kc1, name)), f"K {name}"
    for name in ("codes", "norm"):
        assert torch.equal(getattr(vc, name), getattr(vc1, name)), f"V {name}"
    assert torch.equal(out0, out1)


@pytest.mark.parametrize("kbits,vbits,kbits2,vbits2", [(3, 3, None, None), (3, 3, 2, 2), (4, 4, 3, 3)])
def test_step_against_oracle(kbits, vbits, kbits2, vbits2):
    """The step's output equals the oracle's decode over the oracle-quantized
    context plus the appended token; whole-width, 2.5-bit and 3.5-bit caches."""
    d, bsz, hkv, hq, cap, kind = 128, 2, 2, 8, 512, "rht"
    k, v, rot, qjl, caches, q, knew, vnew = _setup(bsz, hkv, hq, cap, kind, kbits, vbits, seed=70,
                                                   kbits2=kbits2 or 0, vbits2=vbits2 or 0)
    pos_np = np.array([300, 511], dtype=np.int32)
    pos = torch.from_numpy(pos_np).cuda()
    lens_np = pos_np + 1
    lens = torch.from_numpy(lens_np).cuda()
    (kc, vc) = caches[0]
    out = torch.empty((bsz, hq, d), device="cuda")
    ws = B.workspace(B.tq_decode_step_workspace(q, kc, vc, lens, cap, rot, qjl, out, knew, vnew, pos))
    B.tq_decode_step(q, kc, vc, lens, cap, rot, qjl, out, knew, vnew, pos, ws)
    torch.cuda.synchronize()
    # oracle: the context with the new token written at its slot
    k2, v2 = k.copy(), v.copy()
    kn = knew.float().cpu().numpy().reshape(bsz, hkv, d)
    vn = vnew.float().cpu().numpy().reshape(bsz, hkv, d)
    for b in range(bsz):
        k2[b, :, pos_np[b]] = kn[b]
        v2[b, :, pos_np[b]] = vn[b]
    pi, s = P.oracle_mats(d, kind)
    kq = oq.quantize(W.round_bf16(k2).reshape(-1, d).astype(np.float64), pi, "prod", kbits, s, bits2=kbits2)
    vq = oq.quantize(W.round_bf16(v2).reshape(-1, d).astype(np.float64), pi, "mse", vbits, bits2=vbits2)
    sh = (bsz, hkv, cap)
    kcd = {"idx": kq["idx"].reshape(sh + (d,)), "norm16": kq["norm16"].reshape(sh),
           "rnorm16": kq["rnorm16"].reshape(sh), "z": kq["z"].reshape(sh + (d,))}
    vcd = {"idx": vq["idx"].reshape(sh + (d,)), "norm16": vq["norm16"].reshape(sh)}
    want, _ = oa.decode(q.cpu().numpy().astype(np.float64), kcd, vcd, lens_np.tolist(), pi, s,
                        kq["centroids"], vq["centroids"])
    got = out.cpu().numpy()
    # the tolerance is for unit-scale coordinates: scaled by the largest value
    # norm over sqrt(d), as in the full-shape decode test
    scale = np.max(vq["norm16"]) / np.sqrt(d)
    assert np.max(np.abs(got - want)) <= OUT_TOL * scale, np.max(np.abs(got - want)) / scale


def test_step_rejects_bad_args_before_enqueueing():
    d, bsz, hkv, hq, cap = 128, 1, 2, 8, 64
    k, v, rot, qjl, caches, q, knew, vnew = _setup(bsz, hkv, hq, cap, "rht", 3, 3, seed=90)
    (kc, vc) = caches[0]
    before = kc.codes.clone()
    pos = torch.tensor([10], dtype=torch.int32, device="cuda")
    lens = torch.tensor([11], dtype=torch.int32, device="cuda")
    out = torch.empty((bsz, hq, d), device="cuda")
    ws = B.workspace(B.tq_decode_step_workspace(q, kc, vc, lens, cap, rot, qjl, out, knew, vnew, pos))
    with pytest.raises(B.TQError):  # workspace too small: nothing may be enqueued
        B.tq_decode_step(q, kc, vc, lens, cap, rot, qjl, out, knew, vnew, pos, ws[:16])
    torch.cuda.synchronize()
    assert torch.equal(kc.codes, before)


@pytest.mark.parametrize("bsz,hkv,hq,T,kbits,vbits,heavy,samples,kind", [
    # the bench's default line: Llama-3.1-8B decode, 32768 tokens
    (1, 8, 32, 32768, 3, 3, 0.0, [(0, 0), (0, 17), (0, 31)], "rht"),
    # batched decode: 16 sequences of 8192 tokens, both rotations
    (16, 8, 32, 8192, 3, 3, 0.0, [(0, 5), (9, 20), (15, 31)], "rht"),
    (16, 8, 32, 8192, 3, 3, 0.0, [(2, 1), (11, 26), (15, 30)], "dense"),
    # long context: 131072 tokens, 64 q / 8 KV heads, K 3-bit / V 4-bit, 1 % of tokens with norm x 10
    (1, 8, 64, 131072, 3, 4, 0.01, [(0, 3), (0, 62)], "rht"),
])
def test_full_size_step_sampled(bsz, hkv, hq, T, kbits, vbits, heavy, samples, kind):
    """The benchmarked step at the workloads' full shapes and in the bench's
    launch configuration (the new token appended at the last slot of every
    sequence): the appended slots' packed records and sampled query heads
    against the oracle."""
    d = 128
    k, v = W.decode_kv(bsz, hkv, T, seed=5, heavy_frac=heavy)
    rot, qjl = P.handles(d, kind)
    kc = B.Cache("prod", kbits, d, rows=bsz * hkv, capacity=T)
    vc = B.Cache("mse", vbits, d, rows=bsz * hkv, capacity=T)
    # the context up to slot T - 2 comes from the GPU's cache fill; slot T - 1 from the step
    B.tq_quantize_kv(kc, rot, torch.from_numpy(k.reshape(-1, d)).cuda().to(torch.bfloat16), qjl=qjl)
    B.tq_quantize_kv(vc, rot, torch.from_numpy(v.reshape(-1, d)).cuda().to(torch.bfloat16))
    q = torch.from_numpy(W.query_vectors((bsz, hq, d), dtype="bf16", seed=6)).cuda().to(torch.bfloat16)
    knew = torch.from_numpy(W.round_bf16(W.query_vectors((bsz * hkv, d), seed=7) * 2)).cuda().to(torch.bfloat16)
    vnew = torch.from_numpy(W.round_bf16(W.query_vectors((bsz * hkv, d), seed=8))).cuda().to(torch.bfloat16)
    pos = torch.full((bsz,), T - 1, dtype=torch.int32, device="cuda")
    lens = torch.full((bsz,), T, dtype=torch.int32, device="cuda")
    out = torch.empty((bsz, hq, d), device="cuda")
    ws = B.workspace(B.tq_decode_step_workspace(q, kc, vc, lens, T, rot, qjl, out, knew, vnew, pos))
    B.tq_decode_step(q, kc, vc, lens, T, rot, qjl, out, knew, vnew, pos, ws)
    torch.cuda.synchronize()
    got = out.cpu().numpy()

    pi, s = P.oracle_mats(d, kind)
    kn = knew.float().cpu().numpy().reshape(bsz, hkv, d)
    vn = vnew.float().cpu().numpy().reshape(bsz, hkv, d)
    qn = q.float().cpu().numpy()
    # the appended slots: the GPU's packed records against the oracle's quantization of the new tokens
    got_k = P.cache_to_numpy(kc, bsz * hkv * T)
    got_v = P.cache_to_numpy(vc, bsz * hkv * T)
    last = np.arange(bsz * hkv) * T + (T - 1)
    for name, mode, bits, xn, g in (("k", "prod", kbits, kn, got_k), ("v", "mse", vbits, vn, got_v)):
        qz = oq.quantize(xn.reshape(-1, d).astype(np.float64), pi, mode, bits, s if mode == "prod" else None)
        sub = {key: val[last] for key, val in g.items()}
        rep = P.compare_quantized(sub, qz, mode, bits, d, s, label=f"appended-{name}")
        assert rep["code_mismatch"] == 0
    del got_k, got_v
    for b, h in samples:
        kv = h // (hq // hkv)
        kx = k[b, kv].copy()
        vx = v[b, kv].copy()
        kx[T - 1] = kn[b, kv]
        vx[T - 1] = vn[b, kv]
        kq = oq.quantize(W.round_bf16(kx).astype(np.float64), pi, "prod", kbits, s)
        vq = oq.quantize(W.round_bf16(vx).astype(np.float64), pi, "mse", vbits)
        qp, u = oa.query_prep(qn[b, h].astype(np.float64), pi, s)
        lg = oa.key_logits(qp, u, kq["idx"], kq["norm16"], kq["centroids"], kq["rnorm16"], kq["z"], d)
        vhat = vq["norm16"][:, None] * vq["centroids"][vq["idx"]]
        sc = lg / np.sqrt(d)
        pr = np.exp(sc - sc.max())
        pr /= pr.sum()
        want = (pr @ vhat) @ pi
        scale = np.max(vq["norm16"]) / np.sqrt(d)
        err = np.max(np.abs(got[b, h] - want)) / scale
        assert err <= OUT_TOL, (b, h, err)


def test_step_with_pinned_host_io():
    """The step's query, new keys and values and its output may live in pinned
    host memory, which the GPU addresses directly (unified addressing; on a
    Grace-Blackwell node over NVLink-C2C): the kernels read the inputs and
    write the output there, with no copy. Same results, bit for bit, as the
    same step on device buffers."""
    bsz, hkv, hq, cap = 2, 2, 8, 512
    k, v, rot, qjl, caches, q, knew, vnew = _setup(bsz, hkv, hq, cap, "rht", 3, 3, seed=80)
    pos = torch.tensor([200, 511], dtype=torch.int32, device="cuda")
    lens = torch.tensor([201, 512], dtype=torch.int32, device="cuda")
    (kc, vc) = caches[0]
    out0 = torch.empty((bsz, hq, 128), device="cuda")
    ws0 = B.workspace(B.tq_decode_step_workspace(q, kc, vc, lens, cap, rot, qjl, out0, knew, vnew, pos))
    B.tq_decode_step(q, kc, vc, lens, cap, rot, qjl, out0, knew, vnew, pos, ws0)
    (kc1, vc1) = caches[1]
    qh, kh, vh = q.cpu().pin_memory(), knew.cpu().pin_memory(), vnew.cpu().pin_memory()
    outh = torch.full((bsz, hq, 128), float("nan")).pin_memory()
    ws1 = B.workspace(B.tq_decode_step_workspace(qh, kc1, vc1, lens, cap, rot, qjl, outh, kh, vh, pos))
    B.tq_decode_step(qh, kc1, vc1, lens, cap, rot, qjl, outh, kh, vh, pos, ws1)
    torch.cuda.synchronize()
    assert torch.equal(out0.cpu(), outh)
    for name in ("codes", "signs", "norm", "rnorm"):
        assert torch.equal(getattr(kc, name), getattr(kc1, name)), f"K {name}"
    for name in ("codes", "norm"):
        assert torch.equal(getattr(vc, name), getattr(vc1, name)), f"V {name}"


def test_quantized_kv_cache_wrapper_matches_the_calls():
    """QuantizedKVCache.prefill + step equal the tq_quantize_kv / tq_decode_step
    calls they stand for, bit for bit, and the lengths advance by one."""
    d, bsz, hkv, hq, cap, T0 = 128, 2, 2, 8, 256, 100
    k, v = W.decode_kv(bsz, hkv, T0, seed=33)
    kt = torch.from_numpy(k).cuda().to(torch.bfloat16)
    vt = torch.from_numpy(v).cuda().to(torch.bfloat16)
    c = B.QuantizedKVCache(bsz, hq, hkv, cap, d=d, k_bits=3, v_bits=3, rotation="rht")
    c.prefill(kt, vt, [T0, 60])
    # the same through the calls
    kc = B.Cache("prod", 3, d, rows=bsz * hkv, capacity=cap)
    vc = B.Cache("mse", 3, d, rows=bsz * hkv, capacity=cap)
    slots = np.full((bsz, hkv, T0), -1, dtype=np.int64)
    for b, n in enumerate([T0, 60]):
        for h in range(hkv):
            slots[b, h, :n] = (b * hkv + h) * cap + np.arange(n)
    st = torch.from_numpy(slots.reshape(-1)).cuda()
    B.tq_quantize_kv(kc, c.rot, kt.reshape(-1, d), qjl=c.qjl, dst_slot=st)
    B.tq_quantize_kv(vc, c.rot, vt.reshape(-1, d), dst_slot=st)
    lens = torch.tensor([T0, 60], dtype=torch.int32, device="cuda")
    for s in range(3):
        q = torch.from_numpy(W.query_vectors((bsz, hq, d), seed=40 + s)).cuda()
        kn = torch.from_numpy(W.round_bf16(W.query_vectors((bsz, hkv, d), seed=50 + s))).cuda().to(torch.bfloat16)
        vn = torch.from_numpy(W.round_bf16(W.query_vectors((bsz, hkv, d), seed=60 + s))).cuda().to(torch.bfloat16)
        got = c.step(q, kn, vn)
        out = torch.empty((bsz, hq, d), device="cuda")
        new = lens + 1
        ws = B.workspace(B.tq_decode_step_workspace(q, kc, vc, new, cap, c.rot, c.qjl, out,
                                                    kn.reshape(-1, d), vn.reshape(-1, d), lens))
        B.tq_decode_step(q, kc, vc, new, cap, c.rot, c.qjl, out, kn.reshape(-1, d), vn.reshape(-1, d), lens, ws)
        lens = new
        torch.cuda.synchronize()
        assert torch.equal(got, out), s
    assert c.lengths.tolist() == [T0 + 3, 63]
    for name in ("codes", "signs", "norm", "rnorm"):
        assert torch.equal(getattr(c.k, name), getattr(kc, name)), name
    for name in ("codes", "norm"):
        assert torch.equal(getattr(c.v, name), getattr(vc, name)), name


def test_step_captured_in_a_cuda_graph():
    """The step's three launches (the last two programmatic dependents) record
    into a CUDA graph; a replay gives the same cache and output, bit for bit,
    as the same step run eagerly."""
    bsz, hkv, hq, cap = 2, 2, 8, 512
    k, v, rot, qjl, caches, q, knew, vnew = _setup(bsz, hkv, hq, cap, "rht", 3, 3, seed=85)
    pos = torch.tensor([123, 400], dtype=torch.int32, device="cuda")
    lens = torch.tensor([124, 401], dtype=torch.int32, device="cuda")
    (kc, vc) = caches[0]
    out0 = torch.empty((bsz, hq, 128), device="cuda")
    ws0 = B.workspace(B.tq_decode_step_workspace(q, kc, vc, lens, cap, rot, qjl, out0, knew, vnew, pos))
    B.tq_decode_step(q, kc, vc, lens, cap, rot, qjl, out0, knew, vnew, pos, ws0)
    (kc1, vc1) = caches[1]
    out1 = torch.full((bsz, hq, 128), float("nan"), device="cuda")
    ws1 = B.workspace(B.tq_decode_step_workspace(q, kc1, vc1, lens, cap, rot, qjl, out1, knew, vnew, pos))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.tq_decode_step(q, kc1, vc1, lens, cap, rot, qjl, out1, knew, vnew, pos, ws1)
    assert bool(torch.isnan(out1).all())  # captured, not run
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out0, out1)
    for name in ("codes", "signs", "norm", "rnorm"):
        assert torch.equal(getattr(kc, name), getattr(kc1, name)), f"K {name}"
    for name in ("codes", "norm"):
        assert torch.equal(getattr(vc, name), getattr(vc1, name)), f"V {name}"
    assert B.tq_device_errors() == (B.TQ_OK, 0)
