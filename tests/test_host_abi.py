"""CPU tests of the C-ABI library: it loads, exports every symbol the header
declares, its struct layouts match the binding, and its host set-up math
(random stream, rotations, QJL matrix, codebooks) matches the oracle.
No compute call needs a GPU here."""

import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT
from oracle import codebook, rng, rotation


@pytest.fixture(scope="session")
def lib():
    from online_kv_cache_quantize_gb300 import binding, build

    build.build()
    return binding


def _header_functions():
    src = open(os.path.join(ROOT, "include", "tq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(tq_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_symbols_are_exported(lib):
    names = _header_functions()
    assert len(names) >= 20
    cdll = ctypes.CDLL(lib.lib_path())
    for n in names:
        assert hasattr(cdll, n), n
    assert set(names) == set(lib.EXPORTED)


def test_struct_layouts_match(lib):
    lib.load()  # raises on a mismatch


def test_random_stream_matches_oracle(lib):
    assert np.array_equal(lib.tq_random_stream(123, 1000), rng.splitmix64(123, 1000))
    assert np.array_equal(lib.tq_random_stream(5, 10, start=90), rng.splitmix64(5, 10, start=90))


@pytest.mark.parametrize("d,kind", [(16, "dense"), (128, "dense"), (200, "dense"), (64, "rht"), (128, "rht"), (256, "rht")])
def test_rotation_matches_oracle(lib, d, kind):
    r = lib.tq_make_rotation(1, d, kind)
    pi = lib.tq_rotation_get(r)
    assert np.max(np.abs(pi - rotation.make_rotation(1, d, kind))) < 1e-12
    assert np.max(np.abs(pi @ pi.T - np.eye(d))) < 1e-12


def test_qjl_matrix_matches_oracle(lib):
    for m, d in ((128, 128), (200, 200), (64, 128)):
        s = lib.tq_qjl_get(lib.tq_make_qjl(2, m, d))
        want = rng.round_to_bf16(rng.normals(2, m * d).reshape(m, d))
        assert np.array_equal(s, want)


@pytest.mark.parametrize("d", [16, 128, 200])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_codebook_matches_oracle(lib, d, bits):
    c, t = lib.tq_codebook(d, bits)
    co, to = codebook.lloyd_max(d, bits)
    assert np.max(np.abs(c - co)) < 1e-12 and np.max(np.abs(t - to)) < 1e-12
    assert np.array_equal(c, -c[::-1]) and t[len(t) // 2] == 0.0


def test_layout_sizes(lib):
    assert lib.tq_code_bytes(128, 2) == 32 and lib.tq_code_bytes(128, 3) == 48
    assert lib.tq_code_bytes(200, 3) == 80 and lib.tq_code_bytes(200, 1) == 32
    assert lib.tq_sign_bytes(128) == 16 and lib.tq_sign_bytes(200) == 32


def test_two_width_code_stride_matches_oracle(lib):
    """Fractional-rate stride: the packed bit count rounded up to 8 bytes
    (24 / 40 / 56 B for code bits 2/1, 3/2, 4/3 at d = 128), as the oracle's
    packing lays it out; equal widths give the one-width stride."""
    from oracle import quantize as oq
    L = lib.load()
    for cb, cb2, want in ((2, 1, 24), (3, 2, 40), (4, 3, 56)):
        assert L.tq_code_bytes2(128, cb, cb2) == want
        idx = np.zeros((1, 128), dtype=np.int64)
        assert oq.pack_codes(idx, [cb if i % 16 < 8 else cb2 for i in range(128)]).shape[1] == want
    for cb in (1, 2, 3, 4):
        assert L.tq_code_bytes2(128, cb, cb) == L.tq_code_bytes(128, cb)


def test_decode_workspace_plan_on_the_host(lib):
    """The decode plan (no device work): 1 KB of B operands per query row plus
    the split partials, splits of a multiple of 64 tokens; invalid shapes give 0."""
    import ctypes
    L = lib.load()
    a = lib.tq_decode_args()
    a.batch, a.hq, a.hkv, a.d, a.max_seq_len, a.n_splits = 1, 32, 8, 128, 32768, 74
    rows = 32
    chunk = -(-32768 // 74)
    chunk = max(64, -(-chunk // 64) * 64)
    splits = -(-32768 // chunk)
    want = rows * 1024 + rows * splits * (128 + 4) * 4
    assert L.tq_attn_decode_workspace(ctypes.byref(a)) == want
    a.hq = 24  # 24 / 8 = 3 is not a group size
    assert L.tq_attn_decode_workspace(ctypes.byref(a)) == 0
    a.hq, a.d = 32, 96
    assert L.tq_attn_decode_workspace(ctypes.byref(a)) == 0


def test_prefill_workspace_plan_on_the_host(lib):
    """The prefill plan (no device work): q' and u rows plus the split
    partials; invalid shapes give 0."""
    import ctypes
    L = lib.load()
    a = lib.tq_prefill_args()
    a.batch, a.chunk, a.hq, a.hkv, a.d, a.max_context = 1, 512, 32, 8, 128, 32768
    a.k.capacity = 32768
    a.n_splits = 3
    rows = 512 * 32
    want = 2 * rows * 128 * 4 + rows * 3 * (128 + 4) * 4
    assert L.tq_attn_prefill_workspace(ctypes.byref(a)) == want
    a.hq = 12  # 12 / 8 is not a group size
    assert L.tq_attn_prefill_workspace(ctypes.byref(a)) == 0
    a.hq, a.max_context = 32, 40000  # beyond the capacity
    assert L.tq_attn_prefill_workspace(ctypes.byref(a)) == 0
    a.max_context, a.d = 32768, 64
    assert L.tq_attn_prefill_workspace(ctypes.byref(a)) == 0


def test_prefill_stream_k_plan_on_the_host(lib):
    """The tcgen05 prefill's stream-K plan, read through its workspace (q' and
    u rows plus rows x slots partials). 2 units (2 KV heads x one 128-row
    query block) of 8 tiles (1000 tokens) are 16 tiles, at most one per SM,
    so each CTA takes one tile and a unit's rows fill one slot per tile. An
    explicit split count of 3 pads each unit to 3 splits of 3 tiles: three
    slots."""
    import ctypes
    L = lib.load()
    a = lib.tq_prefill_args()
    a.batch, a.chunk, a.hq, a.hkv, a.d, a.max_context = 1, 32, 8, 2, 128, 1000
    a.k.capacity = 1024
    a.k.mode, a.k.bits, a.v.mode, a.v.bits = lib.TQ_PROD, 3, lib.TQ_MSE, 3  # the tcgen05 widths
    rows = 32 * 8

    def want(slots):
        return 2 * rows * 128 * 4 + rows * slots * (128 + 4) * 4

    a.n_splits = 0
    assert L.tq_attn_prefill_workspace(ctypes.byref(a)) == want(8)
    a.n_splits = 3
    assert L.tq_attn_prefill_workspace(ctypes.byref(a)) == want(3)


def test_argument_errors_are_reported(lib):
    with pytest.raises(lib.TQError) as e:
        lib.tq_make_rotation(1, 200, "rht")
    assert "UNSUPPORTED" in str(e.value)
    with pytest.raises(lib.TQError):
        lib.tq_make_rotation(1, 2, "dense")
    with pytest.raises(lib.TQError):
        lib.tq_codebook(128, 5)
    with pytest.raises(lib.TQError):
        lib.tq_make_qjl(1, 0, 128)
    L = lib.load()
    assert L.tq_quantize_kv(None, None) == 1  # TQ_ERR_INVALID_ARG
    assert L.tq_attn_decode(None, None, 0, None) == 1
    assert L.tq_score_topk(None, None, 0, None) == 1
    assert L.tq_attn_decode_workspace(None) == 0
    assert L.tq_attn_prefill(None, None, 0, None) == 1
    assert L.tq_attn_prefill_workspace(None) == 0


@pytest.mark.parametrize("level", [1, 2, 3, 5, 7, 8])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_polar_codebook_matches_oracle(lib, level, bits):
    """The library's PolarQuant angle codebooks (its own quadrature) against
    the oracle's (incomplete-beta masses, Gauss-Legendre moments)."""
    from oracle import polar
    c, t = lib.tq_polar_codebook(level, bits)
    co, to = polar.codebook(level, bits)
    assert np.max(np.abs(c - co)) < 1e-12 and np.max(np.abs(t - to)) < 1e-12
    if level >= 2:
        assert np.max(np.abs(c + c[::-1] - np.pi / 2)) < 1e-13


def test_polar_code_bytes(lib):
    """64 bits1 + 63 bits2 bits at d = 128, rounded up to 16 bytes (the
    oracle's packing of a row gives the same stride); invalid arguments 0."""
    from oracle import polar
    for b1, b2 in ((4, 2), (3, 2), (2, 2), (4, 3), (1, 1), (4, 4), (2, 1)):
        want = polar.pack([np.zeros((1, n), dtype=np.int64) for n in polar.angle_count(128)], 128, b1, b2).shape[1]
        assert lib.tq_polar_code_bytes(128, b1, b2) == want
    assert lib.tq_polar_code_bytes(128, 4, 2) == 48
    assert lib.tq_polar_code_bytes(100, 4, 2) == 0 and lib.tq_polar_code_bytes(128, 5, 2) == 0
    with pytest.raises(lib.TQError):
        lib.tq_polar_codebook(9, 2)
    with pytest.raises(lib.TQError):
        lib.tq_polar_codebook(2, 0)
