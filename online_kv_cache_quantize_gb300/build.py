"""Builds libtq.so in-tree: nvcc for the CUDA sources (sm_103a only), g++ for
the host set-up code, translation units compiled in parallel.

    python -m online_kv_cache_quantize_gb300.build [--force] [--ptxas-verbose]
"""

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtq.so")

CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]
# -ffp-contract=off: the host set-up math rounds the same on x86-64 and
# aarch64 (no fused multiply-adds where the source has none)
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-ffp-contract=off", "-Wall", "-Wextra", "-Wno-unused-parameter"]


def _sources():
    cu = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    cpp = sorted(f for f in os.listdir(CSRC) if f.endswith(".cpp"))
    return cu, cpp


def _headers_mtime():
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    paths.append(os.path.join(os.path.dirname(PKG), "include", "tq.h"))
    return max(os.path.getmtime(p) for p in paths if os.path.exists(p))


def _compile(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("compile failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(force=False, ptxas_verbose=False, jobs=None):
    """Compile and link libtq.so if any source is newer than it. Returns its path."""
    cu, cpp = _sources()
    srcs = [os.path.join(CSRC, f) for f in cu + cpp]
    newest = max([_headers_mtime()] + [os.path.getmtime(s) for s in srcs])
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest and not ptxas_verbose:
        return LIB
    if shutil.which(NVCC) is None and not os.path.exists(NVCC):
        raise RuntimeError("nvcc not found at " + NVCC)
    os.makedirs(BUILD, exist_ok=True)
    include = ["-I", os.path.join(os.path.dirname(PKG), "include"), "-I", CSRC]
    cmds, objs = [], []
    for f in cu:
        obj = os.path.join(BUILD, f + ".o")
        extra = ["-Xptxas", "-v"] if ptxas_verbose else []
        cmds.append([NVCC] + NVCC_FLAGS + extra + include + ["-c", os.path.join(CSRC, f), "-o", obj])
        objs.append(obj)
    for f in cpp:
        obj = os.path.join(BUILD, f + ".o")
        cmds.append(["g++"] + CXX_FLAGS + include + ["-c", os.path.join(CSRC, f), "-o", obj])
        objs.append(obj)
    jobs = jobs or min(len(cmds), os.cpu_count() or 4)
    logs = []
    with cf.ThreadPoolExecutor(jobs) as ex:
        for out in ex.map(_compile, cmds):
            logs.append(out)
    tmp = LIB + ".tmp"
    _compile([NVCC] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"])
    os.replace(tmp, LIB)
    if ptxas_verbose:
        sys.stdout.write("\n".join(l for l in logs if l))
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, ptxas_verbose=a.ptxas_verbose))
