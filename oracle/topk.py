"""Inner-product vector search scored from the codes, fp64 oracle.

What the write-ups say: the same quantizer serves nearest-neighbour search;
on GloVe (d = 200) it reaches better top-k recall than product quantization
without dataset-specific codebooks (A2A TurboQuant explainer, "Benchmarks and
real-world performance", last paragraph; "Applications", vector databases).

Readings: the search estimator is the unbiased PROD one (the MSE one is also
offered); queries are not quantized; the score of database row t for query q
is the logit estimator of the attention oracle; the top k are the k largest
scores, ties broken toward the lower row id.

Pinned by: brute-force full sort on tiny databases; exact top-k on the
originals is reported as recall (a quality figure, not parity).
"""

import numpy as np

from . import attention
from . import quantize as qmod


def scores(queries, pi, s_matrix, idx, norm16, centroids, rnorm16=None, z=None):
    """[Q, N] estimated inner products. PROD when z is given, MSE otherwise."""
    queries = np.atleast_2d(np.asarray(queries, dtype=np.float64))
    qp, u = attention.query_prep(queries, pi, s_matrix)
    # the logit estimator of attention.key_logits, for all queries at once
    base = centroids[idx] @ qp.T
    if z is not None:
        m = np.asarray(s_matrix).shape[0]
        pm = 2.0 * z.astype(np.float64) - 1.0
        base = base + qmod.qjl_scale(m) * rnorm16[:, None] * (pm @ u.T)
    return (norm16[:, None] * base).T


def topk(score_matrix, k):
    """Per row: ids of the k largest scores, ties -> lower id; and their scores."""
    score_matrix = np.atleast_2d(score_matrix)
    q, n = score_matrix.shape
    k = min(k, n)
    ids = np.empty((q, k), dtype=np.int64)
    for i in range(q):
        order = np.lexsort((np.arange(n), -score_matrix[i]))
        ids[i] = order[:k]
    return ids, np.take_along_axis(score_matrix, ids, axis=1)


def exact_topk(queries, database, k):
    """Top-k by the exact inner product on the original vectors (for recall)."""
    s = np.atleast_2d(np.asarray(queries, dtype=np.float64)) @ np.asarray(database, dtype=np.float64).T
    return topk(s, k)


def recall_at_k(found, truth):
    found = np.atleast_2d(found)
    truth = np.atleast_2d(truth)
    hits = [len(set(f.tolist()) & set(t.tolist())) for f, t in zip(found, truth)]
    return float(np.sum(hits)) / truth.size
