"""GPU parity of quantize-on-append against the fp64 oracle, through the C ABI."""

import numpy as np
import pytest
import torch

import parity_util as P
from oracle import quantize as oq
from online_kv_cache_quantize_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from online_kv_cache_quantize_gb300 import build
    build.build()


def _run(x, mode, bits, d, kind, dtype, label, m=None, bits2=None):
    xin = np.asarray(x, dtype=np.float32)
    if dtype == torch.bfloat16:
        xin = W.round_bf16(xin)
    cache = P.gpu_quantize(xin, mode, bits, d, kind, dtype=dtype, m=m, bits2=bits2)
    got = P.cache_to_numpy(cache, xin.shape[0])
    pi, s = P.oracle_mats(d, kind, m)
    qz = oq.quantize(xin.astype(np.float64), pi, mode, bits, s if mode == "prod" else None, bits2=bits2)
    return P.compare_quantized(got, qz, mode, bits, d, s, label=label, bits2=bits2)


def test_outlier_keys_dense_prod3_fp32():
    """4096 x 128 fp32 keys with 4 outlier channels x20, dense QR, 3-bit PROD."""
    x, _ = W.outlier_keys(4096, 128)
    rep = _run(x, "prod", 3, 128, "dense", torch.float32, "outlier_keys")
    assert rep["code_mismatch"] == 0


@pytest.mark.parametrize("kind", ["rht", "dense"])
@pytest.mark.parametrize("mode,bits", [("prod", 3), ("prod", 4), ("mse", 3), ("mse", 4), ("prod", 2), ("mse", 2)])
def test_decode_shaped_bf16(kind, mode, bits):
    k, v = W.decode_kv(1, 2, 1500, heavy_frac=0.01)
    x = (k if mode == "prod" else v).reshape(-1, 128)
    _run(x, mode, bits, 128, kind, torch.bfloat16, f"{kind}-{mode}{bits}")


@pytest.mark.parametrize("mode,bits", [("mse", 1), ("prod", 5), ("mse", 4)])
def test_bit_width_extremes(mode, bits):
    x = np.random.default_rng(3).standard_normal((777, 128)).astype(np.float32)
    _run(x, mode, bits, 128, "rht", torch.float32, f"{mode}{bits}")


@pytest.mark.parametrize("mode,bits", [("prod", 2), ("prod", 4), ("mse", 4)])
def test_d200_dense_mixture(mode, bits):
    db, _ = W.mixture_vectors(3000, d=200)
    _run(db, mode, bits, 200, "dense", torch.float32, f"d200-{mode}{bits}")


@pytest.mark.parametrize("d,kind", [(64, "rht"), (256, "rht"), (64, "dense"), (256, "dense"), (96, "dense")])
def test_other_head_sizes(d, kind):
    x = np.random.default_rng(d).standard_normal((515, d)).astype(np.float32) * 3
    _run(x, "prod", 3, d, kind, torch.float32, f"d{d}-{kind}")


def test_edge_vectors():
    """Zero vector, a huge-norm vector (fp16 saturation), one-hot and tiny values."""
    d = 128
    x = np.zeros((6, d), dtype=np.float32)
    x[1] = 1e4                      # norm 1.13e5 -> saturates to 65504
    x[2, 7] = 1.0                   # one-hot
    x[3] = 1e-30                    # tiny but nonzero
    x[4] = np.random.default_rng(0).standard_normal(d)
    x[5, :] = -2.0
    for kind in ("dense", "rht"):
        _run(x, "prod", 3, d, kind, torch.float32, f"edge-{kind}")
        _run(x, "mse", 4, d, kind, torch.float32, f"edge-{kind}-mse")


@pytest.mark.parametrize("kind", ["dense", "rht"])
@pytest.mark.parametrize("mode,bits", [("prod", 3), ("mse", 3)])
def test_fp16_norm_midpoints(kind, mode, bits):
    """Norms exactly halfway between two fp16 values in some rows of a tile and
    not in the others: the fp64 re-rounding runs for part of a warp's rows and
    must give the ties-to-even fp16 of the exact norm."""
    d = 128
    x = np.random.default_rng(17).standard_normal((48, d)).astype(np.float32)
    # one-hot rows: the norm is the entry, a halfway point with 12 significant
    # bits (the third rounds up to its even neighbour, the others down)
    onehot = [1.0 + 2.0 ** -11, 2049.0, 1.0 + 3 * 2.0 ** -11, 0.5 + 2.0 ** -12]
    # two-entry rows (a, b) with a^2 + b^2 = c^2 exactly in fp32 and c a
    # halfway point; a != b, so no rotated coordinate cancels to a tie at 0
    pairs = [(1995.0, 476.0, 2051.0), (1475.0, 1428.0, 2053.0),
             (1995.0 / 2048, 476.0 / 2048, 2051.0 / 2048), (1475.0 / 4096, 1428.0 / 4096, 2053.0 / 4096)]
    planted, want_n = [0, 5, 9, 16, 30, 33, 40, 47], []
    for k, r in enumerate(planted):
        x[r] = 0.0
        if k % 2 == 0:
            x[r, (7 * k) % d] = onehot[k // 2]
            want_n.append(onehot[k // 2])
        else:
            a, b, c = pairs[k // 2]
            x[r, 11 + k] = a
            x[r, 70 + k] = -b
            want_n.append(c)
    cache = P.gpu_quantize(x, mode, bits, d, kind, dtype=torch.float32)
    got = P.cache_to_numpy(cache, x.shape[0])
    pi, s = P.oracle_mats(d, kind, None)
    qz = oq.quantize(x.astype(np.float64), pi, mode, bits, s if mode == "prod" else None)
    rows = np.array(planted)
    assert np.array_equal(qz["n"][rows], np.array(want_n))
    assert np.array_equal(got["norm"][rows], qz["norm16"][rows]), "ties-to-even fp16 norm"
    rep = P.compare_quantized(got, qz, mode, bits, d, s, label=f"fp16-mid-{kind}-{mode}{bits}")
    assert rep["code_mismatch"] == 0


@pytest.mark.parametrize("n", [1, 2, 31, 33, 64, 65, 100])
def test_ragged_counts(n):
    x = np.random.default_rng(n).standard_normal((n, 128)).astype(np.float32)
    _run(x, "prod", 4, 128, "rht", torch.float32, f"n{n}")


def test_slot_modes_append_and_scatter():
    """append_pos and dst_slot write exactly the addressed slots."""
    d, rows, cap = 128, 6, 40
    rot, qjl = P.handles(d, "rht")
    from online_kv_cache_quantize_gb300 import binding as B
    x = np.random.default_rng(9).standard_normal((rows, d)).astype(np.float32)
    xt = torch.from_numpy(x).cuda()
    cache = B.Cache("prod", 3, d, rows=rows, capacity=cap)
    pos = torch.tensor([5, 39, 0], dtype=torch.int32, device="cuda")  # batch 3 x heads 2
    B.tq_quantize_kv(cache, rot, xt, qjl=qjl, append_pos=pos, heads=2)
    ref = B.Cache("prod", 3, d, rows=1, capacity=rows)
    B.tq_quantize_kv(ref, rot, xt, qjl=qjl)
    slots = torch.tensor([0 * cap + 5, 1 * cap + 5, 2 * cap + 39, 3 * cap + 39, 4 * cap + 0, 5 * cap + 0],
                         device="cuda", dtype=torch.int64)
    torch.cuda.synchronize()
    assert torch.equal(cache.codes[slots], ref.codes)
    assert torch.equal(cache.signs[slots], ref.signs)
    assert torch.equal(cache.norm[slots], ref.norm)
    mask = torch.ones(rows * cap, dtype=torch.bool, device="cuda")
    mask[slots] = False
    assert int(cache.codes[mask].abs().sum()) == 0
    # scatter with one out-of-range slot (skipped)
    cache2 = B.Cache("prod", 3, d, rows=1, capacity=10)
    dst = torch.tensor([9, 0, 3, 100, -1, 4], dtype=torch.int64, device="cuda")
    B.tq_quantize_kv(cache2, rot, xt, qjl=qjl, dst_slot=dst)
    torch.cuda.synchronize()
    for i, sl in enumerate([9, 0, 3, None, None, 4]):
        if sl is not None:
            assert torch.equal(cache2.codes[sl], ref.codes[i])


def test_full_size_prefill_sampled():
    """Full batched-decode prefill shape (16 x 8 heads x 8192 tokens, K and V),
    quantized on the GPU in one call each; sampled rows checked against the oracle."""
    from online_kv_cache_quantize_gb300 import binding as B
    d = 128
    rot, qjl = P.handles(d, "rht")
    k, v = W.decode_kv(16, 8, 8192)
    pi, s = P.oracle_mats(d, "rht")
    rng = np.random.default_rng(1)
    for name, x, mode in (("K", k, "prod"), ("V", v, "mse")):
        xf = x.reshape(-1, d)
        xt = torch.from_numpy(xf).cuda().to(torch.bfloat16)
        cache = B.Cache(mode, 3, d, rows=16 * 8, capacity=8192)
        B.tq_quantize_kv(cache, rot, xt, qjl=qjl if mode == "prod" else None)
        torch.cuda.synchronize()
        rows = np.sort(rng.choice(xf.shape[0], 4096, replace=False))
        got = {key: val[rows] for key, val in P.cache_to_numpy(cache).items()}
        qz = oq.quantize(xf[rows].astype(np.float64), pi, mode, 3, s if mode == "prod" else None)
        P.compare_quantized(got, qz, mode, 3, d, s, label=f"prefill-{name}")


@pytest.mark.parametrize("kind", ["rht", "dense"])
@pytest.mark.parametrize("mode,bits", [("prod", 3), ("prod", 4), ("prod", 5), ("mse", 2), ("mse", 3), ("mse", 4)])
def test_two_width_caches(kind, mode, bits):
    """Fractional rates (2.5 / 3.5 bits per channel): coordinates with
    i % 16 < 8 at `bits`, the rest at `bits - 1`, each group with its own
    codebook, codes packed in coordinate order with an 8-byte stride. 1400
    vectors: the tensor-core kernel."""
    k, v = W.decode_kv(1, 2, 700, heavy_frac=0.01)
    x = (k if mode == "prod" else v).reshape(-1, 128)
    _run(x, mode, bits, 128, kind, torch.bfloat16, f"{kind}-{mode}{bits}/{bits - 1}", bits2=bits - 1)


@pytest.mark.parametrize("n,dtype", [(200, torch.bfloat16), (1000, torch.float32), (4133, torch.bfloat16)])
def test_two_width_sizes_and_dtypes(n, dtype):
    """Two-width caches through the CTA-per-vector kernel (200 vectors), fp32
    input on the dense rotation, and a ragged multi-CTA size."""
    x = np.random.default_rng(n).standard_normal((n, 128)).astype(np.float32) * 2
    kind = "dense" if dtype == torch.float32 else "rht"
    _run(x, "prod", 4, 128, kind, dtype, f"two-width n={n}", bits2=3)
    _run(x, "mse", 3, 128, kind, dtype, f"two-width n={n}", bits2=2)


def test_two_width_rejections():
    rot, qjl = P.handles(128, "rht")
    from online_kv_cache_quantize_gb300 import binding as B
    x = torch.zeros((4, 128), device="cuda")
    bad = B.Cache("mse", 4, 128, rows=1, capacity=4, bits2=2)  # only bits2 = bits - 1
    with pytest.raises(B.TQError):
        B.tq_quantize_kv(bad, rot, x)
