"""Builds libmuon_ns.so in-tree with nvcc for sm_103a.

Usage: python -m newton_schulz_07_gb300.build  (or call build()).
Each translation unit is compiled by its own nvcc process, in parallel, into
_build/ at the repository root; the shared library is linked next to this file.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmuon_ns.so")

SOURCES = ["muon_ns.cu", "gemm_sym.cu", "gemm_full.cu", "gemm_f32.cu", "gemm_wout.cu", "gemm_wout_grp.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    return p.returncode, " ".join(cmd), p.stdout


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, extra_flags=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "muon_ns.h"))
    jobs = []
    objs = []
    for src in SOURCES:
        srcp = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [srcp] + headers):
            jobs.append([nvcc()] + NVCC_FLAGS + list(extra_flags) + ["-c", srcp, "-o", obj])
    with ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        results = list(ex.map(_run, jobs))
    for rc, cmd, out in results:
        if verbose or rc != 0:
            sys.stdout.write(f"$ {cmd}\n{out}")
        if rc != 0:
            raise RuntimeError(f"nvcc failed: {cmd}\n{out}")
    if force or jobs or _stale(LIB, objs):
        rc, cmd, out = _run([nvcc()] + ARCH + ["-shared", "-o", LIB] + objs)
        if verbose or rc != 0:
            sys.stdout.write(f"$ {cmd}\n{out}")
        if rc != 0:
            raise RuntimeError(f"link failed: {cmd}\n{out}")
    return LIB


if __name__ == "__main__":
    build(verbose=True, force="--force" in sys.argv,
          extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else ())
