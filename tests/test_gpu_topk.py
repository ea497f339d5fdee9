"""GPU parity of the inner-product top-k search against the fp64 oracle."""

import numpy as np
import pytest
import torch

import parity_util as P
from oracle import quantize as oq
from oracle import topk as ot
from online_kv_cache_quantize_gb300 import binding as B
from online_kv_cache_quantize_gb300 import workloads as W

pytestmark = pytest.mark.gpu
TIE_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    from online_kv_cache_quantize_gb300 import build
    build.build()


def _gpu_topk(queries, db_cache, n_db, rot, qjl, k):
    qt = torch.from_numpy(np.ascontiguousarray(queries, dtype=np.float32)).cuda()
    ids = torch.full((queries.shape[0], k), -1, dtype=torch.int32, device="cuda")
    sc = torch.zeros((queries.shape[0], k), dtype=torch.float32, device="cuda")
    ws = B.workspace(B.tq_score_topk_workspace(qt, db_cache, n_db, rot, qjl, k, ids, sc))
    B.tq_score_topk(qt, db_cache, n_db, rot, qjl, k, ids, sc, ws)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), sc.cpu().numpy()


def _check_topk(gids, gsc, want_scores, k):
    """ids exact modulo ties: a GPU id may differ only where its oracle score
    ties (within TIE_TOL * scale) the oracle's k-th score; scores within 1e-4."""
    wid, wsc = ot.topk(want_scores, k)
    for i in range(gids.shape[0]):
        scale = max(np.max(np.abs(want_scores[i])), 1e-30)
        kth = wsc[i, -1]
        for j in range(k):
            if gids[i, j] != wid[i, j]:
                s_g = want_scores[i, gids[i, j]]
                assert abs(s_g - kth) <= TIE_TOL * scale or abs(s_g - wsc[i, j]) <= TIE_TOL * scale, (i, j)
        assert np.max(np.abs(gsc[i] - want_scores[i, gids[i]])) <= 1e-4 * scale
        assert len(set(gids[i].tolist())) == k


@pytest.mark.parametrize("mode,bits", [("prod", 2), ("prod", 4), ("mse", 2), ("mse", 4)])
def test_topk_on_oracle_codes(mode, bits):
    d, n = 200, 20000
    db, qs = W.mixture_vectors(n, d=d, queries=37)
    pi, s = P.oracle_mats(d, "dense")
    qz = oq.quantize(db.astype(np.float64), pi, mode, bits, s if mode == "prod" else None)
    cache = P.oracle_cache_planes(qz, mode, bits, 1, n)
    rot, qjl = P.handles(d, "dense")
    gids, gsc = _gpu_topk(qs, cache, n, rot, qjl if mode == "prod" else None, 10)
    want = ot.scores(qs, pi, s if mode == "prod" else None, qz["idx"], qz["norm16"], qz["centroids"],
                     qz.get("rnorm16"), qz.get("z"))
    _check_topk(gids, gsc, want, 10)


def test_topk_exact_ties_prefer_lower_id():
    """Duplicate database rows give exactly equal scores: the lower id comes first."""
    d, n = 128, 5000
    r = np.random.default_rng(4)
    db = r.standard_normal((n, d)).astype(np.float32)
    db[4000:4010] = db[10]           # exact duplicates of row 10
    q = db[10:11] * 3
    pi, s = P.oracle_mats(d, "rht")
    qz = oq.quantize(db.astype(np.float64), pi, "prod", 3, s)
    cache = P.oracle_cache_planes(qz, "prod", 3, 1, n)
    rot, qjl = P.handles(d, "rht")
    gids, _ = _gpu_topk(q, cache, n, rot, qjl, 11)
    assert gids[0].tolist() == [10] + list(range(4000, 4010))


def test_full_size_search_sampled():
    """1e6 x 200 database quantized on the GPU (dense QR, 2-bit PROD); 24
    sampled queries' top-10 checked against the oracle's scores."""
    d, n = 200, 1_000_000
    db, qs = W.mixture_vectors(n, d=d, queries=24)
    rot, qjl = P.handles(d, "dense")
    cache = B.Cache("prod", 2, d, rows=1, capacity=n)
    B.tq_quantize_kv(cache, rot, torch.from_numpy(db).cuda(), qjl=qjl)
    gids, gsc = _gpu_topk(qs, cache, n, rot, qjl, 10)
    pi, s = P.oracle_mats(d, "dense")
    want = np.empty((qs.shape[0], n))
    step = 50_000
    for a in range(0, n, step):  # the oracle in slices to bound host memory
        qz = oq.quantize(db[a:a + step].astype(np.float64), pi, "prod", 2, s)
        want[:, a:a + step] = ot.scores(qs, pi, s, qz["idx"], qz["norm16"], qz["centroids"], qz["rnorm16"], qz["z"])
    _check_topk(gids, gsc, want, 10)
    # quality figure only (not parity): overlap with the exact top-10
    truth, _ = ot.exact_topk(qs, db, 10)
    print(f"recall@10 vs exact inner product, 2-bit PROD, 1e6 rows: {ot.recall_at_k(gids, truth):.3f}")


@pytest.mark.parametrize("mode,bits", [("prod", 2), ("mse", 4), ("prod", 4)])
def test_topk_tensor_core_and_simt_paths(mode, bits):
    """The tcgen05 scan (used for d <= 256) and the SIMT scan rank the same
    scores: both checked against the oracle on the same oracle-packed codes."""
    d, n = 200, 9000  # 9000 rows: two full 4096-row chunks and a ragged one
    db, qs = W.mixture_vectors(n, d=d, queries=45)  # 45 queries: a full and a ragged 32-query block
    pi, s = P.oracle_mats(d, "dense")
    qz = oq.quantize(db.astype(np.float64), pi, mode, bits, s if mode == "prod" else None)
    cache = P.oracle_cache_planes(qz, mode, bits, 1, n)
    rot, qjl = P.handles(d, "dense")
    want = ot.scores(qs, pi, s if mode == "prod" else None, qz["idx"], qz["norm16"], qz["centroids"],
                     qz.get("rnorm16"), qz.get("z"))
    lib = B.load()
    results = {}
    for simt in (0, 1):
        prev = lib.tq_topk_force_simt(simt)
        try:
            results[simt] = _gpu_topk(qs, cache, n, rot, qjl if mode == "prod" else None, 10)
        finally:
            lib.tq_topk_force_simt(prev)
        _check_topk(results[simt][0], results[simt][1], want, 10)
    assert B.tq_device_errors() == (B.TQ_OK, 0)


def test_topk_wide_codes_fall_back():
    """d = 256 with 4-bit codes and 256 sign bits does not fit the tensor-core
    scan's shared-memory plan; the SIMT scan serves it with the same parity."""
    d, n = 256, 3000
    r = np.random.default_rng(12)
    db = r.standard_normal((n, d)).astype(np.float32)
    qs = r.standard_normal((7, d)).astype(np.float32)
    pi, s = P.oracle_mats(d, "rht")
    qz = oq.quantize(db.astype(np.float64), pi, "prod", 5, s)
    cache = P.oracle_cache_planes(qz, "prod", 5, 1, n)
    rot, qjl = P.handles(d, "rht")
    gids, gsc = _gpu_topk(qs, cache, n, rot, qjl, 10)
    want = ot.scores(qs, pi, s, qz["idx"], qz["norm16"], qz["centroids"], qz["rnorm16"], qz["z"])
    _check_topk(gids, gsc, want, 10)
