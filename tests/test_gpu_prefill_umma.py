"""The tcgen05 chunked-prefill scan (keys at PROD 2 / 3 bits or the 3 / 2
fractional rate): against the fp64 oracle, and against the mma.sync scan on
the same oracle-packed caches, over shapes that exercise its tiling: several
128-row query blocks with a ragged last one, 128-token tiles with a ragged
tail, many tiles per split (the 3-deep copy ring wraps many times), splits
that see no token at all, stream-K CTAs whose tile range crosses from one
unit (batch row, KV head, query block) into the next, and repeated runs.

Tolerances: both scans are checked against the oracle at the decode output
tolerance (1e-3 of max nV / sqrt(d)). Against each other they differ only by
fp32 summation order and by where the fp16 hi/lo limbs of q', kappa u and
p nV round (the same limbs, formed in the same precision), so they agree to
1e-4 of that scale, as the one-token prefill agrees with decode.
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
PAIR_TOL = 1e-4


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


def _run(q, gk, gv, q_start, max_context, kind, n_splits=0, mma_sync=False):
    bsz, c, hq, d = q.shape
    lib = B.load()
    prev = lib.tq_prefill_force_mma_sync(1 if mma_sync else 0)
    try:
        rot, qjl = P.handles(d, kind)
        qt = torch.from_numpy(np.ascontiguousarray(q, dtype=np.float32)).cuda()
        qs = torch.tensor(q_start, dtype=torch.int32, device="cuda")
        out = torch.full((bsz, c, hq, d), float("nan"), dtype=torch.float32, device="cuda")
        ws = B.workspace(B.tq_attn_prefill_workspace(qt, gk, gv, qs, max_context, rot, qjl, out, n_splits=n_splits))
        B.tq_attn_prefill(qt, gk, gv, qs, max_context, rot, qjl, out, ws, n_splits=n_splits)
        torch.cuda.synchronize()
    finally:
        lib.tq_prefill_force_mma_sync(prev)
    _, flags = B.tq_device_errors(reset=True)
    assert flags == 0, f"device error word {flags:#x}"
    return out.cpu().numpy()


def _scale(vc):
    return max(np.max(vc["norm16"]) / np.sqrt(128), 1e-30)


@pytest.mark.parametrize("kind", ["rht", "dense"])
@pytest.mark.parametrize("kbits,vbits", [(3, 3), (2, 4), (3, 1), (2, 2)])
def test_umma_prefill_against_oracle_and_mma_sync(kind, kbits, vbits):
    """Batch 2, 12 q / 3 KV heads (G = 4), a 45-token chunk = 180 rows per KV
    head (a full 128-row CTA and a ragged one), context 1000 / 700 (128-token
    tiles with ragged tails), automatic splits; outlier data."""
    k, v = W.decode_kv(2, 3, 1024, heavy_frac=0.05, seed=40 + kbits * 5 + vbits)
    kc, vc, gk, gv, kq, vq, pi, s = _caches(k, v, kbits, vbits, kind)
    q = W.query_vectors((2, 45, 12, 128), seed=41)
    q_start = [955, 655]
    new = _run(q, gk, gv, q_start, 1000, kind)
    old = _run(q, gk, gv, q_start, 1000, kind, mma_sync=True)
    want = oa.prefill(q.astype(np.float64), kc, vc, q_start, pi, s, kq["centroids"], vq["centroids"])
    sc = _scale(vc)
    assert np.max(np.abs(new - want)) <= OUT_TOL * sc
    assert np.max(np.abs(new - old)) <= PAIR_TOL * sc


def test_umma_prefill_many_tiles_per_split_and_repeatable():
    """One split over 4096 slots: 32 tiles through the 3-deep ring in one CTA
    (the barrier phases wrap many times); two runs are bit-identical; the
    automatic split plan gives the same output within summation order."""
    k, v = W.decode_kv(1, 2, 4096, heavy_frac=0.01, seed=50)
    kc, vc, gk, gv, kq, vq, pi, s = _caches(k, v, 3, 3, "rht")
    q = W.query_vectors((1, 33, 8, 128), dtype="bf16", seed=51)
    q_start = [4096 - 33]
    a = _run(q, gk, gv, q_start, 4096, "rht", n_splits=1)
    b = _run(q, gk, gv, q_start, 4096, "rht", n_splits=1)
    assert np.array_equal(a, b)
    c = _run(q, gk, gv, q_start, 4096, "rht")
    sc = _scale(vc)
    assert np.max(np.abs(a - c)) <= 1e-5 * sc
    want = oa.prefill(q.astype(np.float64), kc, vc, q_start, pi, s, kq["centroids"], vq["centroids"])
    assert np.max(np.abs(a - want)) <= OUT_TOL * sc


def test_umma_prefill_first_chunk_empty_splits():
    """A 200-token chunk at position 0 with 8 splits of 128 slots over a
    1024-slot context: row blocks whose last token is early see only the
    first splits (the others have no tile and write empty partials); the
    causal triangle falls inside tiles."""
    k, v = W.decode_kv(1, 2, 1024, seed=52)
    kc, vc, gk, gv, kq, vq, pi, s = _caches(k, v, 2, 3, "dense")
    q = W.query_vectors((1, 200, 4, 128), seed=53)
    out = _run(q, gk, gv, [0], 1024, "dense", n_splits=8)
    want = oa.prefill(q.astype(np.float64), kc, vc, [0], pi, s, kq["centroids"], vq["centroids"])
    assert np.max(np.abs(out - want)) <= OUT_TOL * _scale(vc)


@pytest.mark.parametrize("vbits", [2, 3, 4])
def test_umma_prefill_fractional_rates(vbits):
    """Keys at 3 / 2 PROD bits (2 / 1 code bits in two channel groups) with
    fractional values 2/1, 3/2, 4/3, against the oracle and mma.sync."""
    k, v = W.decode_kv(1, 2, 768, heavy_frac=0.05, seed=60 + vbits)
    kc, vc, gk, gv, kq, vq, pi, s = _caches(k, v, 3, vbits, "rht", kbits2=2, vbits2=vbits - 1)
    q = W.query_vectors((1, 40, 8, 128), seed=61)
    new = _run(q, gk, gv, [700], 740, "rht")
    old = _run(q, gk, gv, [700], 740, "rht", mma_sync=True)
    want = oa.prefill(q.astype(np.float64), kc, vc, [700], pi, s, kq["centroids"], vq["centroids"])
    sc = _scale(vc)
    assert np.max(np.abs(new - want)) <= OUT_TOL * sc
    assert np.max(np.abs(new - old)) <= PAIR_TOL * sc


def test_query_prep_unaligned_view_matches():
    """The tensor-core query prep (RHT) reads q as 16-byte vectors; a query
    view that is only 4-byte aligned takes the row kernel instead. Both give
    the same output within fp32 summation order (u = S q' summed in a
    different order), and both match the oracle."""
    k, v = W.decode_kv(1, 2, 512, seed=70)
    kc, vc, gk, gv, kq, vq, pi, s = _caches(k, v, 3, 3, "rht")
    q = W.query_vectors((1, 24, 8, 128), seed=71)
    aligned = _run(q, gk, gv, [480], 504, "rht")
    rot, qjl = P.handles(128, "rht")
    flat = torch.empty(q.size + 1, dtype=torch.float32, device="cuda")
    qv = flat[1:].view(q.shape)  # 4-byte aligned only
    qv.copy_(torch.from_numpy(np.ascontiguousarray(q, dtype=np.float32)))
    assert qv.data_ptr() % 16 == 4
    qs = torch.tensor([480], dtype=torch.int32, device="cuda")
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    ws = B.workspace(B.tq_attn_prefill_workspace(qv, gk, gv, qs, 504, rot, qjl, out))
    B.tq_attn_prefill(qv, gk, gv, qs, 504, rot, qjl, out, ws)
    torch.cuda.synchronize()
    unaligned = out.cpu().numpy()
    sc = _scale(vc)
    assert np.max(np.abs(aligned - unaligned)) <= 1e-5 * sc
    want = oa.prefill(q.astype(np.float64), kc, vc, [480], pi, s, kq["centroids"], vq["centroids"])
    assert np.max(np.abs(unaligned - want)) <= OUT_TOL * sc


def test_umma_prefill_stream_k_segments_cross_units():
    """Stream-K: 2 batch rows x 4 KV heads x one 128-row query block (64
    chunk tokens, G = 2) = 8 units of 25 tiles each (3200 tokens), so 200
    tiles over at most one CTA per SM. Each CTA takes 2 tiles, so some start
    in one unit and end in the next, and a unit's rows fill up to 13 partial
    slots. The second row's chunk sits at 1500, so most of its units' tiles
    lie past the causal limit: those segments have no tile and write empty
    partials. Checked against the oracle and the mma.sync scan."""
    k, v = W.decode_kv(2, 4, 3200, heavy_frac=0.02, seed=80)
    kc, vc, gk, gv, kq, vq, pi, s = _caches(k, v, 3, 3, "rht")
    q = W.query_vectors((2, 64, 8, 128), seed=81)
    q_start = [3136, 1500]
    new = _run(q, gk, gv, q_start, 3200, "rht")
    old = _run(q, gk, gv, q_start, 3200, "rht", mma_sync=True)
    want = oa.prefill(q.astype(np.float64), kc, vc, q_start, pi, s, kq["centroids"], vq["centroids"])
    sc = _scale(vc)
    assert np.max(np.abs(new - want)) <= OUT_TOL * sc
    assert np.max(np.abs(new - old)) <= PAIR_TOL * sc
