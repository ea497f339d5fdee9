"""tq_attn_decode_static, the decode entry point that allocates nothing.

Callers that may not allocate device memory at decode time (an engine plugin
whose host owns all device memory, work enqueued during CUDA graph capture, a
runtime that forbids allocation after start-up) use this entry point; its
scratch is an array inside the library. Its output must match the
workspace-taking tq_attn_decode on the same inputs, call after call, since the
array is shared and keeps the previous call's contents.
"""

import numpy as np
import pytest
import torch

import parity_util as P
from online_kv_cache_quantize_gb300 import binding as B
from online_kv_cache_quantize_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_static_scratch_decode_matches_workspace_decode():
    from online_kv_cache_quantize_gb300 import build
    build.build()
    d, bsz, hkv, hq, cap = 128, 2, 4, 16, 1024
    k, v = W.decode_kv(bsz, hkv, cap)
    rot, qjl = P.handles(d, "rht")
    kc = B.Cache("prod", 3, d, rows=bsz * hkv, capacity=cap)
    vc = B.Cache("mse", 3, d, rows=bsz * hkv, capacity=cap)
    B.tq_quantize_kv(kc, rot, torch.from_numpy(k.reshape(-1, d)).cuda().to(torch.bfloat16), qjl=qjl)
    B.tq_quantize_kv(vc, rot, torch.from_numpy(v.reshape(-1, d)).cuda().to(torch.bfloat16))
    # two calls in a row with different queries; the second call has shorter
    # sequences and fewer splits, so partials the first call left in the
    # shared array would show up in its output if it read any of them
    calls = [(11, [cap, 777], 0), (12, [300, 65], 2)]
    for call, (seed, lens_list, splits) in enumerate(calls):
        lens = torch.tensor(lens_list, dtype=torch.int32, device="cuda")
        q = torch.from_numpy(W.query_vectors((bsz, hq, d), seed=seed)).cuda()
        ref = torch.empty((bsz, hq, d), dtype=torch.float32, device="cuda")
        ws = B.workspace(B.tq_attn_decode_workspace(q, kc, vc, lens, cap, rot, qjl, ref, n_splits=splits))
        B.tq_attn_decode(q, kc, vc, lens, cap, rot, qjl, ref, ws, n_splits=splits)
        got = torch.full((bsz, hq, d), float("nan"), dtype=torch.float32, device="cuda")
        B.tq_attn_decode_static(q, kc, vc, lens, cap, rot, qjl, got, n_splits=splits)
        torch.cuda.synchronize()
        # the same kernels on the same inputs with a deterministic split
        # count and merge order: bit-identical, not merely close
        assert torch.equal(got, ref), f"call {call}: max |static - workspace| = {float((got - ref).abs().max())}"


def test_static_scratch_passes_argument_errors_through():
    from online_kv_cache_quantize_gb300 import build
    build.build()
    d, bsz, hkv, hq, cap = 128, 1, 2, 6, 64
    rot, qjl = P.handles(d, "rht")
    kc = B.Cache("prod", 3, d, rows=bsz * hkv, capacity=cap)
    vc = B.Cache("mse", 3, d, rows=bsz * hkv, capacity=cap)
    q = torch.zeros((bsz, hq, d), device="cuda")
    out = torch.zeros((bsz, hq, d), device="cuda")
    lens = torch.full((bsz,), cap, dtype=torch.int32, device="cuda")
    # group size 3 is not built: the same status as tq_attn_decode
    for fn in (lambda: B.tq_attn_decode_static(q, kc, vc, lens, cap, rot, qjl, out),
               lambda: B.tq_attn_decode(q, kc, vc, lens, cap, rot, qjl, out, B.workspace(1 << 20))):
        with pytest.raises(B.TQError) as e:
            fn()
        assert e.value.status == B.TQ_ERR_UNSUPPORTED, str(e.value)


def test_static_scratch_rejects_oversized_arguments():
    from online_kv_cache_quantize_gb300 import build
    build.build()
    d, bsz, hkv, hq, cap = 128, 8, 32, 256, 2048
    rot, qjl = P.handles(d, "rht")
    # 2048 query rows x 32 splits x 132 floats = 35 MB of scratch: more than the array holds
    kc = B.Cache("prod", 3, d, rows=bsz * hkv, capacity=cap)
    vc = B.Cache("mse", 3, d, rows=bsz * hkv, capacity=cap)
    q = torch.zeros((bsz, hq, d), device="cuda")
    out = torch.zeros((bsz, hq, d), device="cuda")
    lens = torch.full((bsz,), cap, dtype=torch.int32, device="cuda")
    assert B.tq_attn_decode_workspace(q, kc, vc, lens, cap, rot, qjl, out, n_splits=32) > (8 << 20)
    with pytest.raises(B.TQError) as e:
        B.tq_attn_decode_static(q, kc, vc, lens, cap, rot, qjl, out, n_splits=32)
    assert "WORKSPACE" in str(e.value)
