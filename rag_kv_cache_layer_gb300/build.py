"""Builds libcacheblend.so in-tree with nvcc for sm_103a.

Each CUDA translation unit compiles in parallel into ``_build/``; the shared
library is linked next to this file.  Usage: ``python -m
rag_kv_cache_layer_gb300.build`` (or ``build()`` from Python).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libcacheblend.so")

SOURCES = [
    "cb_api.cu",
    "k_rope.cu",
    "k_select.cu",
    "k_rows.cu",
    "k_gemm_simt.cu",
    "k_gemm_tc.cu",
    "k_gemm_sab.cu",
    "k_attn_simt.cu",
    "k_attn_tc.cu",
    "k_qprobe.cu",
    "k_noalloc.cu",
]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"),
                 "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-I", os.path.join(ROOT, "include"), "-I", CSRC,
                   "--expt-relaxed-constexpr", *extra]


def _compile(src: str, verbose: bool, extra=()) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *_flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}")
    return obj


def build(verbose: bool = False, ptxas_verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    extra = ("-Xptxas", "-v") if ptxas_verbose else ()
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose or ptxas_verbose, extra),
                           SOURCES))
    tmp = LIB + ".tmp"
    # every symbol must resolve inside the library or its runtime deps
    cmd = [nvcc(), *ARCH, "-shared", "-Xlinker", "--no-undefined", "-o", tmp, *objs, "-lcuda"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("link failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, ptxas_verbose="--ptxas" in sys.argv))
