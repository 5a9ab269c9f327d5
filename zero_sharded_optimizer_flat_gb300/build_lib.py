"""Builds libzopt.so in-tree for sm_103a with nvcc (no cmake): one object per source,
compiled in parallel, then linked with the static CUDA runtime so the library loads on a
machine without a GPU (for the ABI checks) and needs nothing but the driver on a GPU machine.

Usage: python -m zero_sharded_optimizer_flat_gb300.build_lib [--force]
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
BUILD = os.path.join(ROOT, "_build", "zopt")
LIB = os.path.join(PKG, "libzopt.so")

SOURCES = ["common.cpp", "layout.cpp", "norm.cu", "norm_noalloc.cu", "adamw.cu", "rescale.cu", "accum.cu", "ns.cu", "ns_gemm.cu",
           "ns_prep.cu", "ns_fused.cu", "ns_simt.cu", "muon.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _digest() -> str:
    h = hashlib.sha256()
    h.update(" ".join(ARCH + SOURCES).encode())
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            path = os.path.join(d, name)
            if os.path.isfile(path):
                h.update(name.encode())
                with open(path, "rb") as f:
                    h.update(f.read())
    with open(__file__, "rb") as f:
        h.update(f.read())
    return h.hexdigest()


def _compile(src: str) -> str:
    nvcc = _nvcc()
    obj = os.path.join(BUILD, src + ".o")
    path = os.path.join(CSRC, src)
    common = ["-O3", "-std=c++17", f"-I{INCLUDE}", f"-I{CSRC}", "-Xcompiler", "-fPIC,-ffp-contract=off,-fvisibility=hidden"]
    if src.endswith(".cu"):
        cmd = [nvcc, *ARCH, "-lineinfo", *common, "-c", path, "-o", obj]
    else:
        cmd = [nvcc, "-x", "c++", *common, "-c", path, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compiling {src} failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libzopt.so unless it is up to date; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    stamp = os.path.join(BUILD, "stamp")
    digest = _digest()
    if not force and os.path.exists(LIB) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return LIB
    with ThreadPoolExecutor(max_workers=min(8, len(SOURCES))) as ex:
        objs = list(ex.map(_compile, SOURCES))
    tmp = LIB + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"linking libzopt.so failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(digest)
    if verbose:
        print(f"built {LIB}")
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
