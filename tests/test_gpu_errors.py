"""The device error word and the bounded mbarrier wait, on the GPU.

The wait is made to run out without any fault: a self-test kernel waits on an
mbarrier that nothing arrives on, gives up after its limit, sets its bit and
returns; the host reads the bit back and clears it."""

import pytest
import torch

from online_kv_cache_quantize_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from online_kv_cache_quantize_gb300 import build
    build.build()


def test_bounded_wait_runs_out_and_reports():
    B.tq_device_errors(reset=True)
    B.tq_selftest_bounded_wait(2000)  # 2 ms
    st, flags = B.tq_device_errors(reset=True)
    assert st == B.TQ_ERR_TIMEOUT
    assert flags == B.TQ_DEVERR_SELFTEST_WAIT
    st, flags = B.tq_device_errors()
    assert (st, flags) == (B.TQ_OK, 0)
    # the context is still usable
    x = torch.arange(16, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 120.0


def test_selftest_limit_is_validated():
    with pytest.raises(B.TQError):
        B.tq_selftest_bounded_wait(0)
    with pytest.raises(B.TQError):
        B.tq_selftest_bounded_wait(2_000_000)


def test_decode_leaves_the_error_word_clear():
    import numpy as np
    import parity_util as P
    from online_kv_cache_quantize_gb300 import workloads as W
    B.tq_device_errors(reset=True)
    d, hkv, hq, L = 128, 2, 8, 1008
    k, v = W.decode_kv(1, hkv, L)
    rot, qjl = P.handles(d, "rht")
    kc = B.Cache("prod", 3, d, rows=hkv, capacity=L)
    vc = B.Cache("mse", 3, d, rows=hkv, capacity=L)
    B.tq_quantize_kv(kc, rot, torch.from_numpy(k.reshape(-1, d)).cuda().to(torch.bfloat16), qjl=qjl)
    B.tq_quantize_kv(vc, rot, torch.from_numpy(v.reshape(-1, d)).cuda().to(torch.bfloat16))
    q = torch.from_numpy(W.query_vectors((1, hq, d))).cuda()
    lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    out = torch.empty((1, hq, d), dtype=torch.float32, device="cuda")
    ws = B.workspace(B.tq_attn_decode_workspace(q, kc, vc, lens, L, rot, qjl, out))
    B.tq_attn_decode(q, kc, vc, lens, L, rot, qjl, out, ws)
    assert B.tq_device_errors() == (B.TQ_OK, 0)
    assert bool(torch.isfinite(out).all())


@pytest.mark.parametrize("a_in_tmem", [False, True])
@pytest.mark.parametrize("n,k", [(16, 16), (32, 48), (64, 64), (128, 128), (64, 128)])
def test_tcgen05_gemm_matches_cpu(n, k, a_in_tmem):
    """The tcgen05 path (core-matrix smem descriptors, kind::f16 instruction
    descriptor, TMEM accumulators read back with tcgen05.ld; A from shared
    memory or written into TMEM with tcgen05.st) against an exact CPU product:
    small integers, so every sum is exact in fp32."""
    import numpy as np
    rng = np.random.default_rng(n * 1000 + k)
    a = rng.integers(-3, 4, size=(128, k)).astype(np.float16)
    b = rng.integers(-3, 4, size=(n, k)).astype(np.float16)
    want = a.astype(np.float64) @ b.astype(np.float64).T
    B.tq_device_errors(reset=True)
    d = torch.full((128, n), float("nan"), device="cuda")
    B.tq_selftest_umma_gemm(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), d, a_in_tmem=a_in_tmem)
    assert B.tq_device_errors() == (B.TQ_OK, 0)
    assert np.array_equal(d.cpu().numpy().astype(np.float64), want)
