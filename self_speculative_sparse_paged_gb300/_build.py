"""Builds libvegas.so (the Vegas hot-path kernels and their C ABI) in-tree.

nvcc compiles each translation unit for sm_103a in parallel; the verify kernel
source is compiled once per (head_dim, capture) pair so its 28 instantiations
spread over four units.  The library is rebuilt unless the digest stored
beside it matches the current sources, headers, flags and this script (a copied
or stale binary is never trusted on its timestamp).
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libvegas.so")
DIGEST = os.path.join(BUILD, "libvegas.sha256")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE]

UNITS = [
    ("vegas_api.cu", "vegas_api.o", []),
    ("synth.cu", "synth.o", []),
    ("verify_noalloc.cu", "verify_noalloc.o", []),
    ("verify_tc.cu", "verify_tc_d128.o", ["-DVEGAS_TC_D=128"]),
    ("verify_tc.cu", "verify_tc_d64.o", ["-DVEGAS_TC_D=64"]),
    ("select_topk.cu", "select_topk.o", []),
    ("select_window.cu", "select_window.o", []),
    ("raw_aggregate.cu", "raw_aggregate.o", []),
    ("wait_check.cu", "wait_check.o", []),
    ("sparse_decode.cu", "sparse_decode.o", []),
    ("verify_attn.cu", "verify_d128_c1.o", ["-DVEGAS_D=128", "-DVEGAS_CAP=1"]),
    ("verify_attn.cu", "verify_d128_c0.o", ["-DVEGAS_D=128", "-DVEGAS_CAP=0"]),
    ("verify_attn.cu", "verify_d64_c1.o", ["-DVEGAS_D=64", "-DVEGAS_CAP=1"]),
    ("verify_attn.cu", "verify_d64_c0.o", ["-DVEGAS_D=64", "-DVEGAS_CAP=0"]),
]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the Vegas CUDA library cannot be built")
    return cand


def sources_digest() -> str:
    """sha256 over every source and header (name and bytes), the units and
    flags, and this script."""
    h = hashlib.sha256()
    paths = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC))
    paths += sorted(os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE))
    paths.append(os.path.abspath(__file__))
    for p in paths:
        h.update(os.path.basename(p).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(repr((FLAGS, UNITS)).encode())
    return h.hexdigest()


def up_to_date() -> bool:
    if not (os.path.exists(LIB) and os.path.exists(DIGEST)):
        return False
    with open(DIGEST) as f:
        return f.read().strip() == sources_digest()


def build(verbose: bool = False, jobs: int | None = None) -> str:
    """Compile every unit for sm_103a and link libvegas.so; returns its path."""
    if up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    if os.path.exists(DIGEST):
        os.remove(DIGEST)
    cc = nvcc()

    def compile_unit(unit):
        src, obj, extra = unit
        cmd = [cc] + FLAGS + extra + ["-c", os.path.join(CSRC, src), "-o", os.path.join(BUILD, obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} {' '.join(extra)}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stdout.write(f"built {obj}\n")
        return obj

    jobs = jobs or min(len(UNITS), max(1, os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(compile_unit, UNITS))
    tmp = LIB + ".tmp"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + [os.path.join(BUILD, o) for o in objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(DIGEST, "w") as f:
        f.write(sources_digest() + "\n")
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
