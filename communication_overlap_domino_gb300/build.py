"""Builds libdomino_gb300.so in-tree from csrc/ with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into one shared
library with the CUDA runtime linked statically (so the library loads, and
its symbols can be listed, on a machine without a GPU).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import time

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_NAME = "libdomino_gb300.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]
SOURCES = ["api.cu", "gemm.cu", "gemm_pair.cu", "fused.cu", "shard_sum.cu", "noalloc.cu", "plan.cu", "attn.cu", "tensor_peak.cu"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _sources_mtime() -> float:
    latest = 0.0
    for d in (CSRC, INCLUDE):
        for name in os.listdir(d):
            latest = max(latest, os.path.getmtime(os.path.join(d, name)))
    latest = max(latest, os.path.getmtime(os.path.abspath(__file__)))
    return latest


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compiles (if stale) and returns the path of the shared library."""
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= _sources_mtime():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    t0 = time.time()
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc, *ARCH_FLAGS, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if ptxas_verbose:
            cmd += ["-Xptxas", "-v"]
        # export the C-ABI symbols only (they carry default visibility in api.cu)
        procs.append((src, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, cmd, pr in procs:
        out, _ = pr.communicate()
        text = out.decode(errors="replace")
        if pr.returncode != 0:
            failed.append(f"--- {src} ---\n{' '.join(cmd)}\n{text}")
        elif verbose or ptxas_verbose:
            sys.stderr.write(f"--- {src} ---\n{text}")
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = LIB_PATH + ".tmp"
    link = [nvcc, *ARCH_FLAGS, "-shared", "-o", tmp, *objs, "-cudart", "static", "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + " ".join(link) + "\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, LIB_PATH)
    if verbose:
        sys.stderr.write(f"built {LIB_PATH} in {time.time() - t0:.1f}s\n")
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv)
