"""Helpers for the GPU-vs-oracle parity tests (test infrastructure).

Comparison rules (readings of the stated tolerances; see the design notes):
* codes: identical, except a coordinate whose fp64 rotated value lies within
  1e-6 * max(|t_j|, 1/sqrt(d)) of a boundary t_j; such mismatches must stay
  under 1e-5 of all coordinates (plus one, for small cases) and are listed;
* packed bytes: equal to the specification's packing of the GPU's own codes
  (so the layout, padding included, is bit-exact);
* norm: fp16 bits identical except where the fp64 norm is within 1e-6
  (relative) of an fp16 rounding midpoint;
* rnorm and sign bits: a vector with an exempt code mismatch is exempt; else
  fp16(gamma) identical except within GAMMA_WINDOW (relative) of a midpoint,
  and sign bit j identical except where |(S r)_j| <= SIGN_WINDOW *
  ||S_j|| * ||r||. Both windows come from the fp32 error of r.
"""

import numpy as np
import torch

from oracle import codebook as ocb
from oracle import quantize as oq
from oracle import rng as orng
from oracle import rotation as orot
from online_kv_cache_quantize_gb300 import binding as B
from online_kv_cache_quantize_gb300 import workloads as W

CODE_WINDOW = 1e-6
NORM_WINDOW = 1e-6
GAMMA_WINDOW = 2e-5
SIGN_WINDOW = 2e-5


def handles(d, kind, m=None, device=True):
    rot = B.tq_make_rotation(W.ROT_SEED, d, kind)
    qjl = B.tq_make_qjl(W.QJL_SEED, m or d, d)
    if device:
        B.tq_rotation_to_device(rot)
        B.tq_qjl_to_device(qjl)
    return rot, qjl


def oracle_mats(d, kind, m=None):
    pi = orot.make_rotation(W.ROT_SEED, d, kind)
    s = orng.round_to_bf16(orng.normals(W.QJL_SEED, (m or d) * d).reshape(m or d, d))
    return pi, s


def gpu_quantize(x_np, mode, bits, d, kind, dtype=torch.float32, m=None, rot=None, qjl=None, bits2=None):
    """Quantize rows of x on the GPU into a fresh cache (rows=1, capacity=n)."""
    if rot is None:
        rot, qjl = handles(d, kind, m)
    x = torch.from_numpy(np.ascontiguousarray(x_np, dtype=np.float32)).to("cuda").to(dtype)
    n = x.shape[0]
    cache = B.Cache(mode, bits, d, rows=1, capacity=max(n, 1), m=m, bits2=bits2)
    B.tq_quantize_kv(cache, rot, x, qjl=qjl if mode == "prod" else None)
    torch.cuda.synchronize()
    return cache


def cache_to_numpy(cache, n=None):
    n = cache.rows * cache.capacity if n is None else n
    out = {"codes": cache.codes[:n].cpu().numpy(),
           "norm": cache.norm[:n].cpu().numpy().view(np.float16).astype(np.float64)}
    if cache.signs is not None:
        out["signs"] = cache.signs[:n].cpu().numpy()
        out["rnorm"] = cache.rnorm[:n].cpu().numpy().view(np.float16).astype(np.float64)
    return out


def _near_fp16_midpoint(v, rel):
    v = np.abs(np.asarray(v, dtype=np.float64))
    h = oq.fp16_rne(v).astype(np.float16)
    up = np.nextafter(h, np.float16(np.inf)).astype(np.float64)
    dn = np.nextafter(h, np.float16(0)).astype(np.float64)
    hf = h.astype(np.float64)
    mids = np.stack([(hf + up) / 2, (hf + dn) / 2])
    return np.min(np.abs(mids - v[None]), axis=0) <= rel * np.maximum(v, 1e-30)


def compare_quantized(got, qz, mode, bits, d, s_matrix=None, label="", bits2=None):
    """Returns a report dict; raises AssertionError on a parity failure."""
    bp = oq.code_widths(d, mode, bits, bits2)
    n = qz["idx"].shape[0]
    gidx = oq.unpack_codes(got["codes"], d, bp)
    # layout: GPU bytes == spec packing of the GPU's own codes
    assert np.array_equal(oq.pack_codes(gidx, bp), got["codes"]), f"{label}: packed layout differs"
    t = qz["boundaries"]
    win = CODE_WINDOW * np.maximum(np.abs(t), 1 / np.sqrt(d))
    near = np.any(np.abs(qz["y"][..., None] - t) <= win, axis=-1)
    mism = gidx != qz["idx"]
    bad = mism & ~near
    assert not bad.any(), f"{label}: {bad.sum()} code mismatches outside the boundary window, e.g. {np.argwhere(bad)[:5].tolist()}"
    # every exempt mismatch is listed: (row, coordinate, fp64 y, nearest boundary, GPU code, oracle code)
    exempt = []
    for r, i in np.argwhere(mism):
        y = float(qz["y"][r, i])
        trow = t[i] if t.ndim == 2 else t  # a two-group cache has a table per coordinate (NaN-padded)
        trow = trow[np.isfinite(trow)]
        tj = float(trow[np.argmin(np.abs(y - trow))])
        exempt.append((int(r), int(i), y, tj, int(gidx[r, i]), int(qz["idx"][r, i])))
        print(f"{label}: exempt code mismatch row {r} coord {i}: y = {y!r}, boundary {tj!r}, "
              f"|y - t| = {abs(y - tj):.3e}, code gpu {gidx[r, i]} / oracle {qz['idx'][r, i]}")
    assert mism.sum() <= 1e-5 * mism.size + 1, f"{label}: too many exempt code mismatches ({mism.sum()}): {exempt[:10]}"
    exempt_vec = mism.any(axis=1)
    # norm
    nbad = (got["norm"] != qz["norm16"]) & ~_near_fp16_midpoint(qz["n"], NORM_WINDOW)
    assert not nbad.any(), f"{label}: {nbad.sum()} fp16 norms differ, e.g. rows {np.flatnonzero(nbad)[:5].tolist()}"
    rep = {"coords": mism.size, "code_mismatch": int(mism.sum()), "exempt_rows": np.flatnonzero(exempt_vec).tolist(),
           "exempt": exempt}
    if mode == "prod":
        m = s_matrix.shape[0]
        g_ok = (got["rnorm"] == qz["rnorm16"]) | _near_fp16_midpoint(qz["gamma"], GAMMA_WINDOW) | exempt_vec
        assert g_ok.all(), f"{label}: {(~g_ok).sum()} fp16 residual norms differ, e.g. rows {np.flatnonzero(~g_ok)[:5].tolist()}"
        gz = oq.unpack_signs(got["signs"], m)
        assert np.array_equal(oq.pack_signs(gz), got["signs"]), f"{label}: sign layout differs"
        srow = np.linalg.norm(s_matrix, axis=1)
        tol = SIGN_WINDOW * srow[None, :] * qz["gamma"][:, None]
        z_ok = (gz == qz["z"]) | (np.abs(qz["sproj"]) <= tol) | exempt_vec[:, None]
        assert z_ok.all(), f"{label}: {(~z_ok).sum()} sign bits differ, e.g. {np.argwhere(~z_ok)[:5].tolist()}"
        rep["sign_mismatch"] = int((gz != qz["z"]).sum())
        rep["rnorm_mismatch"] = int((got["rnorm"] != qz["rnorm16"]).sum())
    rep["norm_mismatch"] = int((got["norm"] != qz["norm16"]).sum())
    return rep


def oracle_cache_planes(qz, mode, bits, rows, capacity, device="cuda", m=None, bits2=None):
    """Upload the ORACLE's packed planes into a GPU Cache (oracle -> GPU only)."""
    d = qz["idx"].shape[1]
    planes = oq.pack(qz, mode, bits, bits2)
    cache = B.Cache(mode, bits, d, rows=rows, capacity=capacity, m=m, bits2=bits2)
    n = qz["idx"].shape[0]
    assert n == rows * capacity
    cache.codes.copy_(torch.from_numpy(planes["codes"]))
    cache.norm.copy_(torch.from_numpy(planes["norm"].view(np.int16)))
    if mode == "prod":
        cache.signs.copy_(torch.from_numpy(planes["signs"]))
        cache.rnorm.copy_(torch.from_numpy(planes["rnorm"].view(np.int16)))
    return cache


def codebook_of(d, mode, bits):
    return ocb.lloyd_max(d, oq.code_bits(mode, bits))[0]
