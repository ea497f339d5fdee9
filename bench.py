#!/usr/bin/env python
"""Benchmark of the TurboQuant hot path on one GB300 (or N replicas).

One step = one online decode step of a Llama-3.1-8B-shaped layer (batch 1,
32 query / 8 KV heads, d = 128, 32768 cached tokens, randomized-Hadamard
rotation, keys 3-bit PROD, values 3-bit MSE): quantize-on-append of the new
token's K and V for every KV head, then decode attention of all query heads
over the packed cache (query rotation, split-K scan, merge + un-rotation).

Prints one JSON line: value = KV-tokens/s (cached tokens attended per second,
all ranks), with the dominant kernel's roofline, the quantize half's
throughput on the cache fill, an end-to-end figure through the C ABI with
host buffers, the oracle timed on the host cores, and sampled SM clocks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tq|reference]
"""

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attn KV-tokens/s & HBM GB/s (% of GB300 peak); quantize vectors/s"
UNIT = "KV-tokens/s"
WORKLOADS = {
    # the default line: one decode step of a Llama-3.1-8B-shaped layer
    "llama8b_decode_32k": dict(batch=1, hq=32, hkv=8, d=128, seq_len=32768, rotation="rht", k_bits=3, v_bits=3),
    # other decode shapes (parity cases; measured with --workload)
    "batched_decode_16x8k": dict(batch=16, hq=32, hkv=8, d=128, seq_len=8192, rotation="rht", k_bits=3, v_bits=3),
    "long_context_128k": dict(batch=1, hq=64, hkv=8, d=128, seq_len=131072, rotation="rht", k_bits=3, v_bits=4,
                              heavy_frac=0.01),
    # fractional-rate caches (second channel group, coordinates i % 16 >= 8, one bit narrower)
    "llama8b_decode_32k_2p5bit": dict(batch=1, hq=32, hkv=8, d=128, seq_len=32768, rotation="rht", k_bits=3, v_bits=3,
                                      k_bits2=2, v_bits2=2),
    "llama8b_decode_32k_3p5bit": dict(batch=1, hq=32, hkv=8, d=128, seq_len=32768, rotation="rht", k_bits=4, v_bits=4,
                                      k_bits2=3, v_bits2=3),
}
WORKLOAD = dict(name="llama8b_decode_32k", **WORKLOADS["llama8b_decode_32k"])
FLUSH_BYTES = 256 << 20  # > 129 MB L2
SCAN_SOURCES = ["online_kv_cache_quantize_gb300/csrc/decode_mma.cuh", "online_kv_cache_quantize_gb300/csrc/common.cuh",
                "online_kv_cache_quantize_gb300/csrc/pipeline.cuh"]


def _bits(w, kv):
    """'3', or '3/2' for a fractional-rate cache (bits of the two channel groups)."""
    b2 = w.get(kv + "_bits2")
    return f"{w[kv + '_bits']}/{b2}" if b2 else str(w[kv + "_bits"])


def _peaks(key="hbm_gbs"):
    """(peak, source): the measured HBM copy GB/s or cuBLAS bf16 TFLOP/s, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p[key]), "measured"
    except Exception:
        return (6800.0 if key == "hbm_gbs" else 1900.0), "fallback"


def _kernel_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic(name, paths, workload, alg_bytes):
    """Per-launch DRAM bytes from a committed ncu capture, if the kernel source
    is unchanged: as captured on the record's own workload, else scaled to
    this launch by its algorithmic bytes (the scan's traffic grows with the
    cache it reads). Returns (bytes or None, how)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[name]
        if rec["source_hash"] != _kernel_hash(paths):
            return None, "kernel changed since the capture"
        if rec["workload_name"] == workload:
            return rec["dram_bytes_per_launch"], "captured on this workload"
        return (rec["dram_bytes_per_launch"] * alg_bytes / rec["alg_bytes_per_launch"],
                f"scaled from the {rec['workload_name']} capture by algorithmic bytes")
    except Exception:
        return None, "no capture"


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        load = [r for r in rows if (num(r[4]) or 0) > 0] or rows
        sm = [num(r[1]) for r in load if num(r[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in load:
            for n, v in zip(names, r[6:10]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(load[0][2]),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(load)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, device):
    """Element-wise maximum of a list of floats over the ranks of the default
    process group (the slowest rank's times); the values themselves on one rank."""
    import torch
    import torch.distributed as dist

    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(world_size, units_per_step, steps, total_ms):
    """Whole-job units per second: each of world_size replicas processed
    units_per_step per step for `steps` steps in total_ms (the slowest rank's)."""
    return world_size * units_per_step * steps / (total_ms / 1e3)


# --------------------------------------------------------------- tq arm ----
def run_tq(args):
    import torch
    import torch.distributed as dist

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from online_kv_cache_quantize_gb300 import binding as B
    from online_kv_cache_quantize_gb300 import build as bld
    from online_kv_cache_quantize_gb300 import workloads as W

    if rank == 0:
        bld.build()
    if ws > 1:
        dist.barrier()
    L = B.load()
    w = WORKLOAD
    bsz, hq, hkv, d, T = w["batch"], w["hq"], w["hkv"], w["d"], w["seq_len"]
    rows = bsz * hkv
    rot = B.tq_rotation_to_device(B.tq_make_rotation(W.ROT_SEED, d, w["rotation"]))
    qjl = B.tq_qjl_to_device(B.tq_make_qjl(W.QJL_SEED, d, d))
    kx, vx = W.decode_kv(bsz, hkv, T, seed=W.DATA_SEED + rank, heavy_frac=w.get("heavy_frac", 0.0))
    kdev = torch.from_numpy(kx.reshape(-1, d)).cuda().to(torch.bfloat16)
    vdev = torch.from_numpy(vx.reshape(-1, d)).cuda().to(torch.bfloat16)
    del kx, vx
    kc = B.Cache("prod", w["k_bits"], d, rows=rows, capacity=T, bits2=w.get("k_bits2"))
    vc = B.Cache("mse", w["v_bits"], d, rows=rows, capacity=T, bits2=w.get("v_bits2"))
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream

    # --- argument blocks built once (the per-step calls only swap events) ---
    def qargs(cache, x, qj):
        a = B.tq_quant_args()
        a.cache = cache.struct()
        a.rot = rot.handle
        a.qjl = qj.handle if qj is not None else None
        a.x = x.data_ptr()
        a.x_dtype = B.TQ_BF16
        a.x_stride = d
        a.n = x.shape[0]
        return a

    fill_k, fill_v = qargs(kc, kdev, qjl), qargs(vc, vdev, None)
    q = torch.from_numpy(W.query_vectors((bsz, hq, d), dtype="bf16", seed=W.QUERY_SEED + rank)).cuda().to(torch.bfloat16)
    knew = torch.from_numpy(W.query_vectors((rows, d), seed=100 + rank)).cuda().to(torch.bfloat16)
    vnew = torch.from_numpy(W.query_vectors((rows, d), seed=200 + rank)).cuda().to(torch.bfloat16)
    # the step's inputs (query, new key, new value) in one buffer, so that the
    # end-to-end run below moves them with one host-to-device copy
    inbuf = torch.cat([q.reshape(-1), knew.reshape(-1), vnew.reshape(-1)])
    q, knew, vnew = (inbuf[: q.numel()].view(q.shape), inbuf[q.numel(): q.numel() + knew.numel()].view(knew.shape),
                     inbuf[q.numel() + knew.numel():].view(vnew.shape))
    append = torch.full((bsz,), T - 1, dtype=torch.int32, device="cuda")
    lens = torch.full((bsz,), T, dtype=torch.int32, device="cuda")
    out = torch.empty((bsz, hq, d), dtype=torch.float32, device="cuda")
    da, _keep = B._decode_struct(q, kc, vc, lens, T, rot, qjl, out)
    wsz = L.tq_attn_decode_workspace(ctypes.byref(da))
    wsb = B.workspace(wsz)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def check(s, what):
        if s != 0:
            raise RuntimeError(f"{what}: {B.status_name(s)} {L.tq_last_error().decode()}")

    # one decode step through the public API: tq_decode_step appends the new
    # token's K and V and runs the attention, all on the caller's stream
    sa = B.tq_step_args()
    sa.attn = da
    sa.k_new = knew.data_ptr()
    sa.v_new = vnew.data_ptr()
    sa.new_dtype = B.TQ_BF16
    sa.append_pos = append.data_ptr()
    assert L.tq_decode_step_workspace(ctypes.byref(sa)) == wsz

    def step():
        check(L.tq_decode_step(ctypes.byref(sa), wsb.data_ptr(), wsz, sp), "decode step")

    launches_per_step = 3  # query prep with the K and V appends, split-K scan, merge

    # cache fill (quantize all K and V of the context): also the quantize measurement
    check(L.tq_quantize_kv(ctypes.byref(fill_k), sp), "fill K")
    check(L.tq_quantize_kv(ctypes.byref(fill_v), sp), "fill V")
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    # exactly --warmup untimed steps, then (only if asked) a further
    # time-based warm-up, reported separately
    n_warm = 0
    for _ in range(args.warmup):
        flush.fill_(n_warm & 0xFF)
        step()
        n_warm += 1
    torch.cuda.synchronize()
    n_extra, t_warm = 0, time.time()
    while time.time() - t_warm < args.warmup_seconds:
        flush.fill_(n_extra & 0xFF)
        step()
        n_extra += 1
        if n_extra % 256 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()

    # --- quantize measurement: cache fill of the whole context (K and V) ---
    nq_it = 3 if args.quick else 20
    qev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nq_it)]
    for i in range(nq_it):
        flush.fill_(i & 0xFF)
        qev[i][0].record(stream)
        check(L.tq_quantize_kv(ctypes.byref(fill_k), sp), "fill K")
        check(L.tq_quantize_kv(ctypes.byref(fill_v), sp), "fill V")
        qev[i][1].record(stream)
    torch.cuda.synchronize()
    q_ms = statistics.mean(a.elapsed_time(b) for a, b in qev)
    q_vectors = 2 * rows * T
    kbytes = kc.code_stride + B.tq_sign_bytes(d) + 4
    vbytes = vc.code_stride + 2
    q_alg_bytes = rows * T * (2 * d * 2) + rows * T * (kbytes + vbytes)

    # --- the timed region: exactly K steps, L2 flushed between them ---
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    host_s = 0.0
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        h0 = time.perf_counter()
        step()
        host_s += time.perf_counter() - h0
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = sum(step_ms)

    # --- the scan's own launch duration: the same steps again with events the
    # library records around the scan launch on the caller's stream (kept out
    # of the steps above: an event between the launches stops the scan from
    # starting while the query prep still runs) ---
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a_, b_ in sev:  # materialise the raw events so the library can record them
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(i & 0xFF)
        sa.attn.scan_begin = sev[i][0].cuda_event
        sa.attn.scan_end = sev[i][1].cuda_event
        step()
    torch.cuda.synchronize()
    sa.attn.scan_begin = None
    sa.attn.scan_end = None
    scan_ms = [a.elapsed_time(b) for a, b in sev]

    # --- end to end through the C ABI with host buffers (pinned) ---
    ne = 3 if args.quick else max(20, min(K, 200))
    h_in = inbuf.cpu().pin_memory()  # query | new keys | new values, as a caller would stage them
    h_out = torch.empty_like(out, device="cpu").pin_memory()
    # (a) the step on pinned host buffers: its kernels read the query and the
    # new K and V from host memory and write the output there (no copy
    # operations; the bytes cross the CPU-GPU link inside the kernels)
    da_h, _keep_h = B._decode_struct(h_in[: q.numel()].view(q.shape), kc, vc, lens, T, rot, qjl, h_out)
    sa_h = B.tq_step_args()
    sa_h.attn = da_h
    sa_h.k_new = h_in.data_ptr() + q.numel() * 2
    sa_h.v_new = h_in.data_ptr() + (q.numel() + knew.numel()) * 2
    sa_h.new_dtype = B.TQ_BF16
    sa_h.append_pos = append.data_ptr()
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(ne)]
    for i in range(ne):
        flush.fill_(i & 0xFF)
        eev[i][0].record(stream)
        check(L.tq_decode_step(ctypes.byref(sa_h), wsb.data_ptr(), wsz, sp), "decode step (host buffers)")
        eev[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_dev_ms = statistics.mean(a.elapsed_time(b) for a, b in eev)
    # host wall clock per step, as a caller sees it: submit the step, wait
    # for its stream, the output is then readable in pinned host memory; no
    # flush or other work in front of it (so host submission is not hidden)
    h_np = h_out.numpy()  # a host view of the pinned output (the read costs no torch op)
    wall = []
    for i in range(ne):
        h0 = time.perf_counter()
        check(L.tq_decode_step(ctypes.byref(sa_h), wsb.data_ptr(), wsz, sp), "decode step (host buffers)")
        stream.synchronize()
        _ = float(h_np[0, 0, 0])  # the result, read on the host
        wall.append(time.perf_counter() - h0)
    e2e_ms = statistics.mean(wall) * 1e3
    # the same zero-copy step captured once in a CUDA graph and replayed (how a
    # serving loop issues a fixed step: one launch instead of three)
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        check(L.tq_decode_step(ctypes.byref(sa_h), wsb.data_ptr(), wsz, torch.cuda.current_stream().cuda_stream),
              "decode step (graph capture)")
    torch.cuda.synchronize()
    wall = []
    for i in range(ne):
        h0 = time.perf_counter()
        graph.replay()
        stream.synchronize()
        _ = float(h_np[0, 0, 0])
        wall.append(time.perf_counter() - h0)
    e2e_graph_ms = statistics.mean(wall) * 1e3
    del graph
    # (b) the same with explicit copies: host -> device into the step's
    # device buffers, the step, device -> host of the output
    mev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(ne)]
    for i in range(ne):
        flush.fill_(i & 0xFF)
        mev[i][0].record(stream)
        inbuf.copy_(h_in, non_blocking=True)
        step()
        h_out.copy_(out, non_blocking=True)
        mev[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_copy_dev_ms = statistics.mean(a.elapsed_time(b) for a, b in mev)
    wall = []
    for i in range(ne):
        h0 = time.perf_counter()
        inbuf.copy_(h_in, non_blocking=True)
        step()
        h_out.copy_(out, non_blocking=True)
        stream.synchronize()
        _ = float(h_out[0, 0, 0])
        wall.append(time.perf_counter() - h0)
    e2e_copy_ms = statistics.mean(wall) * 1e3
    clocks = sampler.stop()
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_out.numel() * h_out.element_size()

    # the slowest rank's times
    total_ms, e2e_ms, e2e_copy_ms, q_ms, e2e_dev_ms, e2e_copy_dev_ms, e2e_graph_ms = max_over_ranks(
        [total_ms, e2e_ms, e2e_copy_ms, q_ms, e2e_dev_ms, e2e_copy_dev_ms, e2e_graph_ms], "cuda")
    tokens_per_step = bsz * T
    value = job_throughput(ws, tokens_per_step, K, total_ms)

    peak, peak_kind = _peaks()
    # per token: codes (the packed bit count), signs (m = d bits), two fp16
    # norms for K, one for V; plus each query row's B operands
    scan_alg = rows * T * (kc.code_stride + d // 8 + 4 + vc.code_stride + 2) + bsz * hq * 2 * d * 4
    scan_avg_s = statistics.mean(scan_ms) / 1e3
    achieved = scan_alg / scan_avg_s / 1e9
    traffic, traffic_how = _traffic("decode_scan", SCAN_SOURCES, w["name"], scan_alg)
    q_achieved = q_alg_bytes / (q_ms / 1e3) / 1e9
    res = None
    if rank == 0:
        res = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": n_warm,
            "warmup_extra_steps": n_extra,
            "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": w["name"], "batch": bsz, "hq": hq, "hkv": hkv, "d": d, "seq_len": T,
                       "rotation": w["rotation"], "k_bits": w["k_bits"], "v_bits": w["v_bits"],
                       **({"k_bits2": w["k_bits2"], "v_bits2": w["v_bits2"]} if w.get("k_bits2") else {}),
                       "step": "append 1 token per KV head (quantize K and V) + decode attention over seq_len tokens",
                       "l2": "flushed (256 MiB write) before every timed step", "parallelism": f"replicas x{ws}"},
            "hbm_gbs": {"scan": achieved, "quantize": q_achieved},
            "roofline": {"kernel": "decode_mma_kernel (split-K scan)", "bound": "hbm", "achieved": achieved,
                         "peak": peak, "unit": "GB/s", "frac": achieved / peak, "peak_source": peak_kind,
                         "alg_bytes_per_launch": scan_alg, "avg_launch_us": scan_avg_s * 1e6,
                         "traffic": traffic, "traffic_source": traffic_how},
            "quantize": {"vectors_per_s": q_vectors / (q_ms / 1e3), "vectors_per_call": q_vectors,
                         "workload": (f"cache fill: {bsz} x {hkv} KV heads x {T} tokens, K ({_bits(w, 'k')}-bit PROD) "
                                      f"and V ({_bits(w, 'v')}-bit MSE), bf16 in, {w['rotation']}"),
                         "roofline": {"bound": "hbm", "achieved": q_achieved, "peak": peak, "unit": "GB/s",
                                      "frac": q_achieved / peak, "alg_bytes_per_call": q_alg_bytes}},
            "e2e": {"value": job_throughput(ws, tokens_per_step, 1, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": ne, "ms_per_step": e2e_ms,
                    "clock": "host wall clock (time.perf_counter) per step: submit, stream synchronize, output "
                             "read on the host; no flush in front",
                    "transfer": "zero-copy: the step's kernels read the query and the new K and V from pinned host "
                                "memory and write the output to pinned host memory (CPU-GPU link inside the kernels)",
                    "device_events": {"value": job_throughput(ws, tokens_per_step, 1, e2e_dev_ms), "unit": UNIT,
                                      "clock": "CUDA events around the step on its stream, L2 flushed before each"},
                    "graph_replay": {"value": job_throughput(ws, tokens_per_step, 1, e2e_graph_ms), "unit": UNIT,
                                     "ms_per_step": e2e_graph_ms,
                                     "clock": "host wall clock, as above, per replay of the step captured once in "
                                              "a CUDA graph (same zero-copy buffers)"},
                    "with_memcpy": {"value": job_throughput(ws, tokens_per_step, 1, e2e_copy_ms), "unit": UNIT,
                                    "ms_per_step": e2e_copy_ms, "clock": "host wall clock, as above",
                                    "device_events": job_throughput(ws, tokens_per_step, 1, e2e_copy_dev_ms),
                                    "transfer": "cudaMemcpyAsync host->device of the inputs and device->host of "
                                                "the output around the step, on its stream"}},
            "gpu_launches": launches_per_step * K,
            "host_us_per_step": host_s / K * 1e6,
            "clocks": clocks,
        }
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return res


# ----------------------------------------------------- oracle (CPU) arm ----
def oracle_sample(budget_s, w=None):
    """Oracle decode steps on a sample: one KV head and its G query heads over
    `tokens` cached tokens (plus the appended K/V quantize for that head),
    extrapolated linearly to the full step (all KV heads, all tokens)."""
    from oracle import attention as oa
    from oracle import quantize as oq
    from oracle import rng as orng
    from oracle import rotation as orot
    from online_kv_cache_quantize_gb300 import workloads as W

    w = WORKLOAD if w is None else w
    d, T, hkv, hq = w["d"], w["seq_len"], w["hkv"], w["hq"]
    g = hq // hkv
    pi = orot.make_rotation(W.ROT_SEED, d, w["rotation"])
    s = orng.round_to_bf16(orng.normals(W.QJL_SEED, d * d).reshape(d, d))
    k, v = W.decode_kv(1, 1, min(T, 32768), heavy_frac=w.get("heavy_frac", 0.0))
    k, v = k[0, 0].astype(np.float64), v[0, 0].astype(np.float64)
    q = W.query_vectors((g, d), dtype="bf16").astype(np.float64)

    caches = {}

    def cache(tokens):  # the oracle's packed cache of the sample, built untimed
        if tokens not in caches:
            caches[tokens] = (oq.quantize(k[:tokens], pi, "prod", w["k_bits"], s, bits2=w.get("k_bits2")),
                              oq.quantize(v[:tokens], pi, "mse", w["v_bits"], bits2=w.get("v_bits2")))
        return caches[tokens]

    def one(tokens):
        kq, vq = cache(tokens)
        t0 = time.perf_counter()
        # append: quantize the new token's K and V for this KV head
        oq.quantize(k[tokens - 1:tokens], pi, "prod", w["k_bits"], s, bits2=w.get("k_bits2"))
        oq.quantize(v[tokens - 1:tokens], pi, "mse", w["v_bits"], bits2=w.get("v_bits2"))
        for h in range(g):
            qp, u = oa.query_prep(q[h], pi, s)
            lg = oa.key_logits(qp, u, kq["idx"], kq["norm16"], kq["centroids"], kq["rnorm16"], kq["z"], d)
            sc = lg / np.sqrt(d)
            p = np.exp(sc - sc.max())
            p /= p.sum()
            (p @ (vq["norm16"][:, None] * oq.coord_centroids(vq["centroids"], vq["idx"]))) @ pi
        return time.perf_counter() - t0

    probe = 2048
    per_token = min(one(probe) for _ in range(3)) / probe
    tokens = int(max(256, min(T, k.shape[0], budget_s / max(per_token, 1e-9))))
    return one, tokens, hkv


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return None
    cores = len(os.sched_getaffinity(0))
    total_budget = 120.0
    per_step = total_budget / max(1, args.steps + args.warmup)
    one, tokens, hkv = oracle_sample(per_step)
    for _ in range(args.warmup):
        one(tokens)
    times = [one(tokens) for _ in range(args.steps)]
    sample_s = statistics.mean(times)
    full_step_s = sample_s * (WORKLOAD["seq_len"] / tokens) * hkv
    value = WORKLOAD["batch"] * WORKLOAD["seq_len"] / full_step_s
    sample = (f"1 of {hkv} KV heads x {tokens} of {WORKLOAD['seq_len']} tokens per step (K/V quantize + 4-head decode), "
              f"extrapolated linearly to the full step")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": full_step_s * 1e3,
            "ms_per_step_is": "extrapolated from the measured sample (sample_ms_per_step) to the full step",
            "sample_ms_per_step": sample_s * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD["name"], "batch": 1, "hq": WORKLOAD["hq"], "hkv": hkv, "d": 128,
                       "seq_len": WORKLOAD["seq_len"], "rotation": WORKLOAD["rotation"]},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def cpu_baseline_default():
    """The oracle on a bounded sample (about 15 s), for the default run's line."""
    cores = len(os.sched_getaffinity(0))
    one, tokens, hkv = oracle_sample(3.0)
    one(tokens)
    times = [one(tokens) for _ in range(4)]
    full_step_s = statistics.mean(times) * (WORKLOAD["seq_len"] / tokens) * hkv
    return {"value": WORKLOAD["batch"] * WORKLOAD["seq_len"] / full_step_s, "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"4 steps of 1/{hkv} KV heads x {tokens} tokens (quantize + 4-head decode), extrapolated to the full step"}


# ------------------------------------------------------------ search ----
SEARCH = dict(name="vector_search_1m", n_db=1_000_000, nq=10_000, d=200, k=10, rotation="dense")
SEARCH_METRIC = "vector search queries/s (top-10 scored from the codes)"


def run_search(args, mode, bits):
    """Inner-product top-10 over a 1e6 x 200 database quantized on the GPU:
    one step = tq_score_topk for all 1e4 queries. Roofline: the tensor pipe,
    algorithmic 2 * nq * n_db * (d + m) flops per step (m = d for PROD)."""
    import torch
    from online_kv_cache_quantize_gb300 import binding as B
    from online_kv_cache_quantize_gb300 import build as bld
    from online_kv_cache_quantize_gb300 import workloads as W

    torch.cuda.set_device(0)
    bld.build()
    L = B.load()
    w = SEARCH
    n, nq, d, k = w["n_db"], w["nq"], w["d"], w["k"]
    db, qs = W.mixture_vectors(n, d=d, queries=nq)
    rot = B.tq_rotation_to_device(B.tq_make_rotation(W.ROT_SEED, d, w["rotation"]))
    qjl = B.tq_qjl_to_device(B.tq_make_qjl(W.QJL_SEED, d, d)) if mode == "prod" else None
    cache = B.Cache(mode, bits, d, rows=1, capacity=n)
    B.tq_quantize_kv(cache, rot, torch.from_numpy(db).cuda(), qjl=qjl)
    del db
    q = torch.from_numpy(qs).cuda()
    ids = torch.empty((nq, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((nq, k), dtype=torch.float32, device="cuda")
    wsz = B.tq_score_topk_workspace(q, cache, n, rot, qjl, k, ids, sc)
    wsb = B.workspace(wsz)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        B.tq_score_topk(q, cache, n, rot, qjl, k, ids, sc, wsb)

    sampler = ClockSampler(0)
    sampler.start()
    for i in range(args.warmup):
        flush.fill_(i & 0xFF)
        step()
    torch.cuda.synchronize()
    K = max(1, min(args.steps, 10))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in ev]
    # end to end: queries from pinned host memory in, ids and scores out
    hq = torch.from_numpy(qs).pin_memory()
    hids = torch.empty_like(ids, device="cpu").pin_memory()
    hsc = torch.empty_like(sc, device="cpu").pin_memory()
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(3)]
    for i in range(3):
        flush.fill_(i & 0xFF)
        eev[i][0].record(stream)
        q.copy_(hq, non_blocking=True)
        step()
        hids.copy_(ids, non_blocking=True)
        hsc.copy_(sc, non_blocking=True)
        eev[i][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    e2e_ms = statistics.mean(a.elapsed_time(b) for a, b in eev)
    step_s = statistics.mean(ms) / 1e3
    m = d if mode == "prod" else 0
    flops = 2.0 * nq * n * (d + m)
    peak, peak_kind = _peaks("bf16_tflops")
    achieved = flops / step_s / 1e12
    return {
        "metric": SEARCH_METRIC, "value": nq / step_s, "unit": "queries/s", "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 (hi/lo split queries), f32 accumulate", "data": "synthetic",
        "config": {"workload": w["name"], "n_db": n, "nq": nq, "d": d, "k": k, "mode": mode, "bits": bits,
                   "rotation": w["rotation"], "l2": "flushed (256 MiB write) before every timed step"},
        "roofline": {"kernel": "topk_umma_kernel (tcgen05 scan)", "bound": "tensor", "achieved": achieved,
                     "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": peak_kind,
                     "alg_flops_per_step": flops, "traffic": None},
        "e2e": {"value": nq / (e2e_ms / 1e3), "unit": "queries/s", "h2d_bytes_per_step": qs.nbytes,
                "d2h_bytes_per_step": hids.numel() * 4 + hsc.numel() * 4, "steps": 3},
        "gpu_launches": 3 * K,  # query prep, scan, merge
        "clocks": clocks,
        "cpu_baseline": None,
    }


PREFILL = {
    # a 512-token chunk of a Llama-3.1-8B-shaped layer at the end of a 32768-token context
    "llama8b_prefill_512_at_32k": dict(batch=1, chunk=512, hq=32, hkv=8, d=128, context=32768, rotation="rht",
                                       k_bits=3, v_bits=3),
}
PREFILL_METRIC = "chunked-prefill tokens/s (causal attention of the chunk over the packed cache)"


def prefill_oracle_sample(w, budget_s=3.0):
    """The oracle's time per query row of the prefill workload (one KV head's
    prefix quantized untimed, then rows at the chunk's last token timed until
    the budget is spent)."""
    from oracle import attention as oa
    from oracle import quantize as oq
    from online_kv_cache_quantize_gb300 import workloads as W

    d, n = w["d"], w["context"]
    from oracle import rng as orng, rotation as orot

    pi = orot.make_rotation(W.ROT_SEED, d, w["rotation"])
    s = orng.round_to_bf16(orng.normals(W.QJL_SEED, d * d).reshape(d, d))
    k, v = W.decode_kv(1, 1, n)
    kq = oq.quantize(k[0, 0].astype(np.float64), pi, "prod", w["k_bits"], s)
    vq = oq.quantize(v[0, 0].astype(np.float64), pi, "mse", w["v_bits"])
    q = W.query_vectors((8, d), dtype="bf16").astype(np.float64)
    rows, t0 = 0, time.perf_counter()
    while rows < 8 and (rows == 0 or time.perf_counter() - t0 < budget_s):
        qp, u = oa.query_prep(q[rows], pi, s)
        lg = oa.key_logits(qp, u, kq["idx"], kq["norm16"], kq["centroids"], kq["rnorm16"], kq["z"], d)
        sc = lg / np.sqrt(d)
        p = np.exp(sc - sc.max())
        p /= p.sum()
        (p @ (vq["norm16"][:, None] * oq.coord_centroids(vq["centroids"], vq["idx"]))) @ pi
        rows += 1
    return (time.perf_counter() - t0) / rows, rows


def run_prefill(args, name):
    import torch
    from online_kv_cache_quantize_gb300 import binding as B
    from online_kv_cache_quantize_gb300 import build as bld
    from online_kv_cache_quantize_gb300 import workloads as W

    torch.cuda.set_device(0)
    bld.build()
    w = dict(name=name, **PREFILL[name])
    bsz, C, hq, hkv, d, T = w["batch"], w["chunk"], w["hq"], w["hkv"], w["d"], w["context"]
    rot = B.tq_rotation_to_device(B.tq_make_rotation(W.ROT_SEED, d, w["rotation"]))
    qjl = B.tq_qjl_to_device(B.tq_make_qjl(W.QJL_SEED, d, d))
    k, v = W.decode_kv(bsz, hkv, T)
    kc = B.Cache("prod", w["k_bits"], d, rows=bsz * hkv, capacity=T)
    vc = B.Cache("mse", w["v_bits"], d, rows=bsz * hkv, capacity=T)
    B.tq_quantize_kv(kc, rot, torch.from_numpy(k.reshape(-1, d)).cuda().to(torch.bfloat16), qjl=qjl)
    B.tq_quantize_kv(vc, rot, torch.from_numpy(v.reshape(-1, d)).cuda().to(torch.bfloat16))
    del k, v
    qh = torch.from_numpy(W.query_vectors((bsz, C, hq, d), dtype="bf16")).to(torch.bfloat16)
    q = qh.cuda()
    qs = torch.full((bsz,), T - C, dtype=torch.int32, device="cuda")
    out = torch.empty((bsz, C, hq, d), dtype=torch.bfloat16, device="cuda")
    wsb = B.workspace(B.tq_attn_prefill_workspace(q, kc, vc, qs, T, rot, qjl, out))
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        B.tq_attn_prefill(q, kc, vc, qs, T, rot, qjl, out, wsb)

    sampler = ClockSampler(0)
    sampler.start()
    for i in range(args.warmup):
        flush.fill_(i & 0xFF)
        step()
    torch.cuda.synchronize()
    K = max(1, min(args.steps, 20))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    # the scan kernel's own launch duration: the same steps again with events
    # the library records around the scan launch (kept out of the steps above:
    # an event between the launches stops the merge from starting early)
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a_, b_ in sev:  # materialise the raw events so the library can record them
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(i & 0xFF)
        B.tq_attn_prefill(q, kc, vc, qs, T, rot, qjl, out, wsb, scan_events=sev[i])
    torch.cuda.synchronize()
    scan_s = statistics.mean(a.elapsed_time(b) for a, b in sev) / 1e3
    # end to end: the chunk's queries from pinned host memory in, the output out
    qpin = qh.pin_memory()
    opin = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(3)]
    for i in range(3):
        flush.fill_(i & 0xFF)
        eev[i][0].record(stream)
        q.copy_(qpin, non_blocking=True)
        step()
        opin.copy_(out, non_blocking=True)
        eev[i][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    step_s = statistics.mean(a.elapsed_time(b) for a, b in ev) / 1e3
    e2e_s = statistics.mean(a.elapsed_time(b) for a, b in eev) / 1e3
    # per visible (query row, key token) pair: <q', c> (2d), the sign term (2m),
    # the value accumulation (2d)
    pairs = bsz * hq * sum(T - C + i + 1 for i in range(C))
    flops = pairs * 2.0 * (d + d + d)
    peak, peak_kind = _peaks("bf16_tflops")
    achieved = flops / scan_s / 1e12
    res = {
        "metric": PREFILL_METRIC, "value": bsz * C / step_s, "unit": "tokens/s", "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 (hi/lo splits), f32 accumulate", "data": "synthetic",
        "config": {"workload": name, "batch": bsz, "chunk": C, "hq": hq, "hkv": hkv, "d": d, "context": T,
                   "q_start": T - C, "rotation": w["rotation"], "k_bits": w["k_bits"], "v_bits": w["v_bits"],
                   "l2": "flushed (256 MiB write) before every timed step"},
        "roofline": {"kernel": ("prefill_umma_kernel (tcgen05)" if w["k_bits"] <= 3 else "prefill_mma_kernel (mma.sync)"),
                     "bound": "tensor", "achieved": achieved,
                     "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": peak_kind,
                     "alg_flops_per_step": flops, "avg_launch_us": scan_s * 1e6,
                     "step_achieved": flops / step_s / 1e12, "step_frac": flops / step_s / 1e12 / peak,
                     "traffic": None},
        "e2e": {"value": bsz * C / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": qpin.numel() * 2,
                "d2h_bytes_per_step": opin.numel() * 2, "steps": 3},
        "gpu_launches": 3 * K,  # query prep, scan, merge
        "clocks": clocks,
        "cpu_baseline": None,
    }
    if not (args.no_cpu_baseline or args.quick):
        t_row, rows = prefill_oracle_sample(w)
        res["cpu_baseline"] = {"value": 1.0 / (t_row * hq), "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
                               "kind": "oracle",
                               "sample": f"{rows} query rows at the chunk's last token over the {T}-token prefix "
                                         f"of one KV head (prefix quantized untimed); a chunk token is {hq} rows"}
    return res


# ----------------------------------------------------- extra workloads ----
# Every workload line of the hot path's measurement plan, printed inside the
# default JSON line (key "workloads") so that one run records all of them.
EXTRA_DECODE = {
    "llama8b_decode_32k_k4v4": dict(batch=1, hq=32, hkv=8, d=128, seq_len=32768, rotation="rht", k_bits=4, v_bits=4),
    "llama8b_decode_32k_dense": dict(batch=1, hq=32, hkv=8, d=128, seq_len=32768, rotation="dense", k_bits=3,
                                     v_bits=3),
    **{f"batched_decode_16x8k_k{b}v{b}_{rot}": dict(batch=16, hq=32, hkv=8, d=128, seq_len=8192, rotation=rot,
                                                    k_bits=b, v_bits=b)
       for rot in ("rht", "dense") for b in (2, 3, 4)},
    "long_context_128k": WORKLOADS["long_context_128k"],
    "llama8b_decode_32k_2p5bit": WORKLOADS["llama8b_decode_32k_2p5bit"],
    "llama8b_decode_32k_3p5bit": WORKLOADS["llama8b_decode_32k_3p5bit"],
}


def _fill_bytes_per_vector(kc, vc, d):
    """(K, V) packed bytes per token and KV head as the plan counts them:
    codes, m = d sign bits and two fp16 norms for K; codes and one fp16 for V."""
    return kc.code_stride + d // 8 + 4, vc.code_stride + 2


def measure_decode(name, w, K, warmup, flush, data, cpu=True):
    """One decode workload: cache fill (the quantize line), warm-up, K timed
    steps (tq_decode_step, L2 flushed before each), the scan's own events."""
    import torch
    from online_kv_cache_quantize_gb300 import binding as B
    from online_kv_cache_quantize_gb300 import workloads as W

    L = B.load()
    bsz, hq, hkv, d, T = w["batch"], w["hq"], w["hkv"], w["d"], w["seq_len"]
    rows = bsz * hkv
    key = (bsz, hkv, T, w.get("heavy_frac", 0.0))
    if key not in data:
        data.clear()
        torch.cuda.empty_cache()
        kx, vx = W.decode_kv(bsz, hkv, T, heavy_frac=w.get("heavy_frac", 0.0))
        data[key] = (torch.from_numpy(kx.reshape(-1, d)).cuda().to(torch.bfloat16),
                     torch.from_numpy(vx.reshape(-1, d)).cuda().to(torch.bfloat16))
        del kx, vx
    kdev, vdev = data[key]
    rot = B.tq_rotation_to_device(B.tq_make_rotation(W.ROT_SEED, d, w["rotation"]))
    qjl = B.tq_qjl_to_device(B.tq_make_qjl(W.QJL_SEED, d, d))
    kc = B.Cache("prod", w["k_bits"], d, rows=rows, capacity=T, bits2=w.get("k_bits2"))
    vc = B.Cache("mse", w["v_bits"], d, rows=rows, capacity=T, bits2=w.get("v_bits2"))
    stream = torch.cuda.current_stream()
    kb, vb = _fill_bytes_per_vector(kc, vc, d)

    # cache fill = the quantize measurement (K and V of every token)
    qev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(4)]
    for i, (a, b) in enumerate(qev):
        flush.fill_(i & 0xFF)
        a.record(stream)
        B.tq_quantize_kv(kc, rot, kdev, qjl=qjl)
        B.tq_quantize_kv(vc, rot, vdev)
        b.record(stream)
    torch.cuda.synchronize()
    q_ms = statistics.mean(a.elapsed_time(b) for a, b in qev[1:])
    q_alg = rows * T * (2 * d * 2) + rows * T * (kb + vb)

    q = torch.from_numpy(W.query_vectors((bsz, hq, d), dtype="bf16")).cuda().to(torch.bfloat16)
    knew = torch.from_numpy(W.query_vectors((rows, d), seed=100)).cuda().to(torch.bfloat16)
    vnew = torch.from_numpy(W.query_vectors((rows, d), seed=200)).cuda().to(torch.bfloat16)
    append = torch.full((bsz,), T - 1, dtype=torch.int32, device="cuda")
    lens = torch.full((bsz,), T, dtype=torch.int32, device="cuda")
    out = torch.empty((bsz, hq, d), dtype=torch.float32, device="cuda")
    da, _keep = B._decode_struct(q, kc, vc, lens, T, rot, qjl, out)
    sa = B.tq_step_args()
    sa.attn = da
    sa.k_new, sa.v_new, sa.new_dtype, sa.append_pos = knew.data_ptr(), vnew.data_ptr(), B.TQ_BF16, append.data_ptr()
    wsz = L.tq_decode_step_workspace(ctypes.byref(sa))
    wsb = B.workspace(wsz)
    sp = stream.cuda_stream

    def step():
        st = L.tq_decode_step(ctypes.byref(sa), wsb.data_ptr(), wsz, sp)
        if st != 0:
            raise RuntimeError(f"{name}: {B.status_name(st)} {L.tq_last_error().decode()}")

    for i in range(warmup):
        flush.fill_(i & 0xFF)
        step()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a_, b_ in sev:
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(i & 0xFF)
        sa.attn.scan_begin = sev[i][0].cuda_event
        sa.attn.scan_end = sev[i][1].cuda_event
        step()
    torch.cuda.synchronize()
    step_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    scan_s = statistics.mean(a.elapsed_time(b) for a, b in sev) / 1e3
    peak, peak_kind = _peaks()
    scan_alg = rows * T * (kb + vb) + bsz * hq * 2 * d * 4
    achieved = scan_alg / scan_s / 1e9
    traffic, traffic_how = _traffic("decode_scan", SCAN_SOURCES, name, scan_alg)
    q_ach = q_alg / (q_ms / 1e3) / 1e9
    fp16_bytes = rows * T * 2 * d * 2
    res = {
        "value": bsz * T / (step_ms / 1e3), "unit": UNIT, "ms_per_step": step_ms, "steps": K, "warmup": warmup,
        "config": {"workload": name, **{k_: v_ for k_, v_ in w.items()}, "l2": "flushed before every timed step"},
        "roofline": {"kernel": "decode_mma_kernel (split-K scan)", "bound": "hbm", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "peak_source": peak_kind,
                     "alg_bytes_per_launch": scan_alg, "avg_launch_us": scan_s * 1e6, "traffic": traffic,
                     "traffic_source": traffic_how},
        "quantize": {"vectors_per_s": 2 * rows * T / (q_ms / 1e3), "vectors_per_call": 2 * rows * T,
                     "ms_per_call": q_ms,
                     "workload": f"cache fill: K ({_bits(w, 'k')}-bit PROD) and V ({_bits(w, 'v')}-bit MSE), bf16 in",
                     "roofline": {"bound": "hbm", "achieved": q_ach, "peak": peak, "unit": "GB/s",
                                  "frac": q_ach / peak, "alg_bytes_per_call": q_alg}},
        "footprint": {"cache_bytes": rows * T * (kb + vb), "fp16_bytes": fp16_bytes,
                      "ratio_vs_fp16": fp16_bytes / (rows * T * (kb + vb)),
                      "bits_per_value": 8.0 * (kb + vb) / (2 * d)},
        "gpu_launches": 3 * K,
    }
    if w["rotation"] == "dense":
        # the dense rotation's tensor work: 2 d^2 per vector, + 2 m d for keys
        flops = rows * T * (2.0 * d * d) * 2 + rows * T * (2.0 * d * d)
        tpeak, tkind = _peaks("bf16_tflops")
        res["quantize"]["tensor"] = {"alg_flops_per_call": flops, "achieved_tflops": flops / (q_ms / 1e3) / 1e12,
                                     "peak": tpeak, "frac": flops / (q_ms / 1e3) / 1e12 / tpeak}
    if cpu:
        one, tokens, hkv_ = oracle_sample(1.0, w)
        one(tokens)
        t = statistics.mean(one(tokens) for _ in range(2))
        full_s = t * (T / tokens) * hkv_ * bsz
        res["cpu_baseline"] = {"value": bsz * T / full_s, "unit": UNIT, "cores": len(os.sched_getaffinity(0)),
                               "kind": "oracle",
                               "sample": f"2 steps of 1 KV head x {tokens} tokens (quantize + {hq // hkv}-head decode), "
                                         f"extrapolated to {bsz} x {hkv} KV heads x {T} tokens"}
        res["quantize"]["cpu_baseline"] = quantize_cpu_baseline(w)
    del kc, vc
    return res


POLAR = dict(batch=1, hq=32, hkv=8, d=128, seq_len=32768, rotation="rht", k_bits=4, k_bits2=2, v_bits=3)


def measure_polar(name, w, K, warmup, flush, cpu=True):
    """The PolarQuant comparison variant at the 32k decode shape: its key
    quantize (vectors/s) and decode attention over PolarQuant keys and MSE
    values (query prep, polar scan, merge; L2 flushed before each step)."""
    import torch
    from online_kv_cache_quantize_gb300 import binding as B
    from online_kv_cache_quantize_gb300 import workloads as W

    bsz, hq, hkv, d, T = w["batch"], w["hq"], w["hkv"], w["d"], w["seq_len"]
    rows = bsz * hkv
    kx, vx = W.decode_kv(bsz, hkv, T)
    kdev = torch.from_numpy(kx.reshape(-1, d)).cuda().to(torch.bfloat16)
    vdev = torch.from_numpy(vx.reshape(-1, d)).cuda().to(torch.bfloat16)
    del kx, vx
    rot = B.tq_rotation_to_device(B.tq_make_rotation(W.ROT_SEED, d, w["rotation"]))
    kc = B.Cache("polar", w["k_bits"], d, rows=rows, capacity=T, bits2=w["k_bits2"])
    vc = B.Cache("mse", w["v_bits"], d, rows=rows, capacity=T)
    stream = torch.cuda.current_stream()
    qev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(4)]
    for i, (a, b) in enumerate(qev):
        flush.fill_(i & 0xFF)
        a.record(stream)
        B.tq_quantize_kv(kc, rot, kdev)
        b.record(stream)
    B.tq_quantize_kv(vc, rot, vdev)
    torch.cuda.synchronize()
    q_ms = statistics.mean(a.elapsed_time(b) for a, b in qev[1:])
    kb, vb = kc.code_stride + 2, vc.code_stride + 2
    q_alg = rows * T * (2 * d + kb)

    q = torch.from_numpy(W.query_vectors((bsz, hq, d), dtype="bf16")).cuda().to(torch.bfloat16)
    lens = torch.full((bsz,), T, dtype=torch.int32, device="cuda")
    out = torch.empty((bsz, hq, d), dtype=torch.float32, device="cuda")
    da, _keep = B._decode_struct(q, kc, vc, lens, T, rot, None, out)
    L = B.load()
    wsz = L.tq_attn_decode_workspace(ctypes.byref(da))
    wsb = B.workspace(wsz)
    sp = stream.cuda_stream

    def step():
        st = L.tq_attn_decode(ctypes.byref(da), wsb.data_ptr(), wsz, sp)
        if st != 0:
            raise RuntimeError(f"{name}: {B.status_name(st)} {L.tq_last_error().decode()}")

    for i in range(warmup):
        flush.fill_(i & 0xFF)
        step()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a_, b_ in sev:
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(i & 0xFF)
        da.scan_begin = sev[i][0].cuda_event
        da.scan_end = sev[i][1].cuda_event
        step()
    torch.cuda.synchronize()
    da.scan_begin = da.scan_end = None
    step_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    scan_s = statistics.mean(a.elapsed_time(b) for a, b in sev) / 1e3
    peak, peak_kind = _peaks()
    scan_alg = rows * T * (kb + vb) + bsz * hq * d * 4
    achieved = scan_alg / scan_s / 1e9
    q_ach = q_alg / (q_ms / 1e3) / 1e9
    fp16_bytes = rows * T * 2 * d * 2
    res = {
        "value": bsz * T / (step_ms / 1e3), "unit": UNIT, "ms_per_step": step_ms, "steps": K, "warmup": warmup,
        "config": {"workload": name, **w, "keys": "PolarQuant (level-1 angles at k_bits, higher levels at k_bits2)",
                   "step": "decode attention only (query prep, polar scan, merge); the keys are appended by "
                           "tq_quantize_kv", "l2": "flushed before every timed step"},
        "roofline": {"kernel": "polar_decode_kernel (split-K scan)", "bound": "hbm", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak, "peak_source": peak_kind,
                     "alg_bytes_per_launch": scan_alg, "avg_launch_us": scan_s * 1e6, "traffic": None},
        "quantize": {"vectors_per_s": rows * T / (q_ms / 1e3), "vectors_per_call": rows * T, "ms_per_call": q_ms,
                     "workload": f"PolarQuant key fill: {rows} KV heads x {T} tokens, bf16 in",
                     "roofline": {"kernel": "polar_quantize_kernel", "bound": "hbm", "achieved": q_ach, "peak": peak,
                                  "unit": "GB/s", "frac": q_ach / peak, "alg_bytes_per_call": q_alg}},
        "footprint": {"cache_bytes": rows * T * (kb + vb), "fp16_bytes": fp16_bytes,
                      "ratio_vs_fp16": fp16_bytes / (rows * T * (kb + vb))},
        "gpu_launches": 3 * K,
    }
    if cpu:
        res["cpu_baseline"] = polar_cpu_baseline(w)
    del kc, vc, kdev, vdev
    return res


def polar_cpu_baseline(w, tokens=4096):
    """The oracle's PolarQuant decode of one KV head's G query heads over
    `tokens` tokens (keys and values quantized untimed), extrapolated to the
    full step."""
    from oracle import codebook as ocb
    from oracle import polar as op
    from oracle import quantize as oq
    from oracle import rotation as orot
    from online_kv_cache_quantize_gb300 import workloads as W

    d, T, hkv, hq = w["d"], w["seq_len"], w["hkv"], w["hq"]
    g = hq // hkv
    pi = orot.make_rotation(W.ROT_SEED, d, w["rotation"])
    k, v = W.decode_kv(1, 1, tokens)
    kq = op.quantize(k[0, 0].astype(np.float64), pi, w["k_bits"], w["k_bits2"])
    vq = oq.quantize(v[0, 0].astype(np.float64), pi, "mse", w["v_bits"])
    kc = {"packed": op.pack(kq["idx"], d, w["k_bits"], w["k_bits2"])[None, None], "norm16": kq["norm16"][None, None]}
    vcache = {"idx": vq["idx"][None, None], "norm16": vq["norm16"][None, None]}
    q = W.query_vectors((1, g, d), dtype="bf16").astype(np.float64)
    vcent = ocb.lloyd_max(d, w["v_bits"])[0]
    t0 = time.perf_counter()
    op.decode(q, kc, vcache, [tokens], pi, w["k_bits"], w["k_bits2"], vcent)
    dt = time.perf_counter() - t0
    full = dt * (T / tokens) * hkv * w["batch"]
    return {"value": w["batch"] * T / full, "unit": UNIT, "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"1 KV head x {tokens} tokens ({g}-head PolarQuant decode), extrapolated to "
                      f"{w['batch']} x {hkv} KV heads x {T} tokens"}


def quantize_cpu_baseline(w, n=2048):
    """The oracle's quantize of n keys and n values of the workload's law."""
    from oracle import quantize as oq
    from oracle import rng as orng
    from oracle import rotation as orot
    from online_kv_cache_quantize_gb300 import workloads as W

    d = w["d"]
    pi = orot.make_rotation(W.ROT_SEED, d, w["rotation"])
    sm = orng.round_to_bf16(orng.normals(W.QJL_SEED, d * d).reshape(d, d))
    k, v = W.decode_kv(1, 1, n)
    t0 = time.perf_counter()
    oq.quantize(k[0, 0].astype(np.float64), pi, "prod", w["k_bits"], sm, bits2=w.get("k_bits2"))
    oq.quantize(v[0, 0].astype(np.float64), pi, "mse", w["v_bits"], bits2=w.get("v_bits2"))
    dt = time.perf_counter() - t0
    return {"value": 2 * n / dt, "unit": "vectors/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{n} keys + {n} values of the workload's law"}


def search_cpu_baseline(mode, bits, rows=100_000, nq=20):
    """The oracle's scoring + top-10 of nq queries over a `rows`-row slice of
    the database (quantized by the oracle untimed), extrapolated to the full
    search by rows and queries."""
    from oracle import quantize as oq
    from oracle import rng as orng
    from oracle import rotation as orot
    from oracle import topk as otk
    from online_kv_cache_quantize_gb300 import workloads as W

    d = SEARCH["d"]
    db, qs = W.mixture_vectors(rows, d=d, queries=nq)
    pi = orot.make_rotation(W.ROT_SEED, d, SEARCH["rotation"])
    sm = orng.round_to_bf16(orng.normals(W.QJL_SEED, d * d).reshape(d, d)) if mode == "prod" else None
    qz = oq.quantize(db.astype(np.float64), pi, mode, bits, sm)
    t0 = time.perf_counter()
    sc = otk.scores(qs.astype(np.float64), pi, sm, qz["idx"], qz["norm16"], qz["centroids"],
                    qz.get("rnorm16"), qz.get("z") if mode == "prod" else None)
    otk.topk(sc, SEARCH["k"])
    dt = time.perf_counter() - t0
    full = dt * (SEARCH["n_db"] / rows) * (SEARCH["nq"] / nq)
    return {"value": SEARCH["nq"] / full, "unit": "queries/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle", "sample": f"{nq} queries x {rows} database rows, extrapolated to "
                                        f"{SEARCH['nq']} x {SEARCH['n_db']}"}


def run_extra(args):
    """Every other workload line, each with its roofline and its oracle
    baseline on the host cores (bounded samples)."""
    import torch

    out = {}
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    data = {}
    K = max(3, min(args.steps, 20))
    for name, w in EXTRA_DECODE.items():
        try:
            out[name] = measure_decode(name, w, K, max(3, args.warmup), flush, data, cpu=not args.no_cpu_baseline)
        except Exception as e:  # noqa: BLE001 - one failing line must not hide the others
            out[name] = {"error": f"{type(e).__name__}: {e}"}
    data.clear()
    # the prefill quantize of the batched workload: 16 x 8 x 8192 K and V
    for name in ("batched_decode_16x8k_k3v3_rht", "batched_decode_16x8k_k3v3_dense"):
        if "quantize" in out.get(name, {}):
            q = dict(out[name]["quantize"])
            q["workload"] = "prefill quantize-on-append of 16 x 8 KV heads x 8192 tokens, K and V (2,097,152 vectors)"
            out["prefill_quantize_16x8x8k_" + name.rsplit("_", 1)[1]] = q
    for tag in ("prod2", "prod4"):
        try:
            r = run_search(args, tag[:-1], int(tag[-1]))
            if not args.no_cpu_baseline:
                r["cpu_baseline"] = search_cpu_baseline(tag[:-1], int(tag[-1]))
            out["vector_search_1m_" + tag] = r
        except Exception as e:  # noqa: BLE001
            out["vector_search_1m_" + tag] = {"error": f"{type(e).__name__}: {e}"}
    try:
        out["polar_decode_32k_k4k2_v3"] = measure_polar("polar_decode_32k_k4k2_v3", POLAR, K, max(3, args.warmup), flush,
                                                        cpu=not args.no_cpu_baseline)
    except Exception as e:  # noqa: BLE001
        out["polar_decode_32k_k4k2_v3"] = {"error": f"{type(e).__name__}: {e}"}
    try:
        out["llama8b_prefill_512_at_32k"] = run_prefill(args, "llama8b_prefill_512_at_32k")
    except Exception as e:  # noqa: BLE001
        out["llama8b_prefill_512_at_32k"] = {"error": f"{type(e).__name__}: {e}"}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--warmup-seconds", type=float, default=0.0,
                    help="extra time-based warm-up after the --warmup steps (reported as warmup_extra_steps)")
    ap.add_argument("--impl", choices=["tq", "reference"], default="tq")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="only the default decode line (skip the other workload lines)")
    ap.add_argument("--quick", action="store_true", help="short run for profiling: no clock window, no oracle timing")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="llama8b_decode_32k")
    ap.add_argument("--k-bits", type=int, default=None)
    ap.add_argument("--v-bits", type=int, default=None)
    ap.add_argument("--rotation", choices=["rht", "dense"], default=None)
    ap.add_argument("--search", choices=["prod2", "prod4", "mse2", "mse4"], default=None,
                    help="time the 1e6 x 200 inner-product top-10 search instead of the decode step")
    ap.add_argument("--search-rows", type=int, default=None, help="database rows (smaller case for profiling)")
    ap.add_argument("--search-queries", type=int, default=None, help="queries (smaller case for profiling)")
    ap.add_argument("--prefill", choices=sorted(PREFILL), default=None,
                    help="time chunked-prefill attention instead of the decode step")
    ap.add_argument("--prefill-context", type=int, default=None, help="context length (smaller case for profiling)")
    ap.add_argument("--polar", action="store_true",
                    help="time only the PolarQuant line (key quantize and decode over PolarQuant keys)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    WORKLOAD.clear()
    WORKLOAD.update(name=args.workload, **WORKLOADS[args.workload])
    for key, val in (("k_bits", args.k_bits), ("v_bits", args.v_bits), ("rotation", args.rotation)):
        if val is not None:
            WORKLOAD[key] = val
    if args.search:
        if args.search_rows:
            SEARCH["n_db"] = args.search_rows
        if args.search_queries:
            SEARCH["nq"] = args.search_queries
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the search has no reference arm here; "
                              "its oracle parity is in tests/test_gpu_topk.py"}))
            return
        print(json.dumps(run_search(args, args.search[:-1], int(args.search[-1]))), flush=True)
        return
    if args.prefill:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the prefill line has no reference arm here; "
                              "its oracle parity is in tests/test_gpu_prefill.py and its cpu_baseline times the "
                              "oracle"}))
            return
        if args.prefill_context:
            PREFILL[args.prefill]["context"] = args.prefill_context
        print(json.dumps(run_prefill(args, args.prefill)), flush=True)
        return
    if args.polar:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the PolarQuant line has no reference arm here; "
                              "its oracle parity is in tests/test_gpu_polar.py"}))
            return
        import torch
        flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        print(json.dumps(measure_polar("polar_decode_32k_k4k2_v3", POLAR, max(3, args.steps), args.warmup, flush,
                                       cpu=not (args.no_cpu_baseline or args.quick))), flush=True)
        return
    if args.impl == "reference":
        res = run_reference(args)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    ws, rank, _ = _dist()
    res = run_tq(args)
    if rank == 0 and res is not None:
        if ws == 1 and not (args.no_cpu_baseline or args.quick):
            res["cpu_baseline"] = cpu_baseline_default()
        else:
            res["cpu_baseline"] = None
        if ws == 1 and not (args.quick or args.no_extra):
            res["workloads"] = run_extra(args)
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
