"""Seeded synthetic inputs shaped like the write-ups' workloads.

This module holds none of the method's arithmetic: it only draws inputs
(NumPy PCG64) and rounds them to the storage dtype. Both the CUDA path and the
fp64 oracle receive exactly these arrays.

Shapes follow the workloads the write-ups discuss: d = 128 heads of a
Llama-3.1-8B-class model with grouped-query attention (Qiita TurboQuant
article, "Rotate, then quantize", last paragraph), contexts of 8k-128k tokens
(A2A TurboQuant explainer, "The KV-cache bottleneck" and "Benchmarks"), KV
activations with a few outlier channels (Qiita, "Rotate, then quantize"), and
GloVe-like d = 200 vector search (A2A, "Benchmarks"). No dataset or model
weights are used; these draws stand in for them.

Seeds: data 0, rotation 1, QJL projection 2, queries 3.
"""

import numpy as np

DATA_SEED = 0
ROT_SEED = 1
QJL_SEED = 2
QUERY_SEED = 3


def round_bf16(x):
    """float32 -> nearest bfloat16 value (ties to even), returned as float32."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def bf16_bits(x):
    """Upper 16 bits of float32 values that are already bfloat16-exact."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def outlier_keys(n=4096, d=128, n_outliers=4, scale=20.0, seed=DATA_SEED):
    """float32 [n, d] i.i.d. N(0,1) with n_outliers fixed channels scaled by `scale`."""
    rng = np.random.default_rng(seed)
    ch = rng.choice(d, size=n_outliers, replace=False)
    x = rng.standard_normal((n, d)).astype(np.float32)
    x[:, ch] *= np.float32(scale)
    return x, np.sort(ch)


def query_vectors(shape, seed=QUERY_SEED, dtype="f32"):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal(shape).astype(np.float32)
    return round_bf16(q) if dtype == "bf16" else q


def decode_kv(batch, hkv, seq_len, d=128, n_outliers=4, outlier_scale=20.0,
              lognormal_sigma=0.5, heavy_frac=0.0, heavy_scale=10.0, seed=DATA_SEED):
    """K and V as bfloat16-exact float32 arrays [batch, hkv, seq_len, d].

    x = s * (z * w_h): z ~ N(0, I); w_h is 1 except `outlier_scale` on
    n_outliers seeded channels per KV head (drawn separately for K and V);
    s ~ LogNormal(0, sigma) per (token, K/V), shared across heads; a seeded
    `heavy_frac` of tokens has s multiplied by heavy_scale.
    """
    rng = np.random.default_rng(seed)
    out = []
    for _kv in range(2):
        w = np.ones((hkv, d), dtype=np.float32)
        for h in range(hkv):
            ch = rng.choice(d, size=n_outliers, replace=False)
            w[h, ch] = outlier_scale
        s = rng.lognormal(0.0, lognormal_sigma, size=(batch, seq_len)).astype(np.float32)
        if heavy_frac > 0:
            heavy = rng.random((batch, seq_len)) < heavy_frac
            s = np.where(heavy, s * np.float32(heavy_scale), s)
        x = np.empty((batch, hkv, seq_len, d), dtype=np.float32)
        for b in range(batch):
            z = rng.standard_normal((hkv, seq_len, d), dtype=np.float32)
            x[b] = z * w[:, None, :] * s[b][None, :, None]
        out.append(round_bf16(x))
    return out[0], out[1]


def mixture_vectors(n, d=200, components=50, seed=DATA_SEED, queries=0, query_seed=QUERY_SEED):
    """Unit-normalised draws from a Gaussian mixture with anisotropic diagonal covariances.

    Component weights uniform, means ~ N(0, I), per-axis stds exp(U[ln 0.1, ln 1]).
    Returns (database float32 [n, d], queries float32 [queries, d]).
    """
    rng = np.random.default_rng(seed)
    mu = rng.standard_normal((components, d))
    sd = np.exp(rng.uniform(np.log(0.1), 0.0, size=(components, d)))

    def draw(r, count):
        comp = r.integers(0, components, size=count)
        x = mu[comp] + sd[comp] * r.standard_normal((count, d))
        x /= np.linalg.norm(x, axis=1, keepdims=True)
        return x.astype(np.float32)

    db = draw(rng, n)
    qs = draw(np.random.default_rng(query_seed), queries) if queries else np.zeros((0, d), np.float32)
    return db, qs


# Named workloads (sizes as the write-ups' shapes suggest; see the design notes)
WORKLOADS = {
    "outlier_keys_4096x128": dict(kind="keys", n=4096, d=128),
    "llama8b_decode_32k": dict(kind="decode", batch=1, hq=32, hkv=8, seq_len=32768, d=128),
    "batched_decode_16x8k": dict(kind="decode", batch=16, hq=32, hkv=8, seq_len=8192, d=128),
    "long_context_128k": dict(kind="decode", batch=1, hq=64, hkv=8, seq_len=131072, d=128,
                              heavy_frac=0.01),
    "mixture_search_1m_d200": dict(kind="search", n=1_000_000, d=200, queries=10_000),
}
