"""Decode attention scored from the packed codes, fp64 oracle.

What the write-ups say:
* the fused kernel rotates the query once and forms dot products straight
  from the stored indices, with no full de-quantization (A2A TurboQuant
  explainer, end of "Stage 2" and "How to implement", the PyTorch item; the
  pro tip on the pre-rotated query path);
* the residual sign sketch removes the bias of the inner product (Qiita
  TurboQuant article, "One more stage so attention does not break").

The logit of key t for query q (q' = Pi q, u = S q'):
    l_t = n_t * ( <q', cK[idx_t]> + sqrt(pi/2)/m * gamma_t * <u, 2 z_t - 1> )
using the stored float16 n_t and gamma_t. Because Pi is orthogonal,
<q', c[idx]> = <q, Pi^T c[idx]>, and <u, 2z-1> = <q', S^T (2z-1)>, so l_t is
<q, x~_t> for the explicit PROD reconstruction.

Attention (readings: the pages give no softmax scale, mask or output format):
    s_t = scale * l_t, scale = 1/sqrt(d) unless given; all L_b cached tokens
    are visible; p = softmax(s) (exact, max-subtracted, fp64);
    a = sum_t p_t nV_t cV[idxV_t] in the rotated domain; o = Pi^T a.
GQA: query head h reads KV head gqa_map[h], default h // (Hq / Hkv).

Pinned by: with an identity "quantizer" the function reduces to textbook
softmax(q K^T / sqrt(d)) V; the estimator equals <q, x~> computed densely;
the estimator is unbiased over rotation/projection seeds (tests).
"""

import numpy as np

from . import quantize as qmod


def query_prep(q, pi, s_matrix=None):
    """q' = Pi q and, when S is given, u = S q' (rows are query vectors)."""
    qp = np.asarray(q, dtype=np.float64) @ np.asarray(pi).T
    u = None if s_matrix is None else qp @ np.asarray(s_matrix, dtype=np.float64).T
    return qp, u


def key_logits(qprime, u, idx, norm16, centroids, rnorm16=None, z=None, m=None):
    """l_t for one query against T keys. idx [T, d]; z [T, m] bool."""
    base = qmod.coord_centroids(centroids, idx) @ qprime
    if z is not None:
        pm = 2.0 * z.astype(np.float64) - 1.0
        base = base + qmod.qjl_scale(m) * rnorm16 * (pm @ u)
    return norm16 * base


def attention_from_rotated(qprime, khat, vhat, scale, pi):
    """Generic single-head decode from rotated-domain key/value reconstructions.

    l_t = <q', khat_t>; p = softmax(scale * l); a = sum p_t vhat_t; o = Pi^T a.
    """
    logits = khat @ qprime
    s = scale * logits
    s = s - np.max(s)
    p = np.exp(s)
    p = p / np.sum(p)
    a = p @ vhat
    return a @ np.asarray(pi), logits


def default_gqa_map(hq, hkv):
    if hq % hkv:
        raise ValueError("Hq must be a multiple of Hkv for the default GQA map")
    g = hq // hkv
    return np.arange(hq) // g


def decode(q, kcache, vcache, seq_lens, pi, s_matrix, k_centroids, v_centroids,
           scale=None, gqa_map=None):
    """Decode attention over a quantized cache.

    q: [B, Hq, d]. kcache / vcache: dicts of unpacked per-slot arrays indexed
    [B, Hkv, T] (+ coordinate axes): 'idx', 'norm16' and, for keys, 'rnorm16'
    and 'z'. Returns (out [B, Hq, d], logits list [B][Hq] -> [L_b]).
    """
    q = np.asarray(q, dtype=np.float64)
    bsz, hq, d = q.shape
    hkv = kcache["idx"].shape[1]
    m = np.asarray(s_matrix).shape[0]
    if gqa_map is None:
        gqa_map = default_gqa_map(hq, hkv)
    if scale is None or scale == 0:
        scale = 1.0 / np.sqrt(d)
    out = np.zeros((bsz, hq, d))
    logits = [[None] * hq for _ in range(bsz)]
    for b in range(bsz):
        L = int(seq_lens[b])
        for h in range(hq):
            kv = int(gqa_map[h])
            if L == 0:
                continue  # no visible token: output 0 by definition
            qp, u = query_prep(q[b, h], pi, s_matrix)
            l = key_logits(qp, u, kcache["idx"][b, kv, :L], kcache["norm16"][b, kv, :L],
                           k_centroids, kcache["rnorm16"][b, kv, :L], kcache["z"][b, kv, :L], m)
            s = scale * l
            s = s - np.max(s)
            p = np.exp(s)
            p = p / np.sum(p)
            vhat = vcache["norm16"][b, kv, :L, None] * qmod.coord_centroids(v_centroids, vcache["idx"][b, kv, :L])
            a = p @ vhat
            out[b, h] = a @ np.asarray(pi)
            logits[b][h] = l
    return out, logits


def prefill(q, kcache, vcache, q_start, pi, s_matrix, k_centroids, v_centroids, scale=None, gqa_map=None):
    """Chunked-prefill attention over a quantized cache (causal).

    Readings (the write-ups give decode only; prefill is the other shape of
    the same attention, over 32k-128k contexts): q [B, C, Hq, d] holds the
    queries of C consecutive tokens of each sequence, the first at position
    q_start[b]; the cache already holds those tokens' keys and values (the
    chunk is quantized on append like every other token), and query i of
    sequence b sees slots 0 .. q_start[b] + i (a causal mask), capped at the
    cache's capacity. Each query is therefore one decode over its visible
    prefix; this is written as exactly that.

    Returns out [B, C, Hq, d].
    """
    q = np.asarray(q, dtype=np.float64)
    bsz, c, hq, d = q.shape
    cap = kcache["idx"].shape[2]
    out = np.zeros((bsz, c, hq, d))
    for i in range(c):
        lens = [min(max(int(q_start[b]) + i + 1, 0), cap) for b in range(bsz)]
        out[:, i], _ = decode(q[:, i], kcache, vcache, lens, pi, s_matrix, k_centroids, v_centroids,
                              scale=scale, gqa_map=gqa_map)
    return out
