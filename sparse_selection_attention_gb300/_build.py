"""In-tree build of the QSA CUDA library (sm_103a) with plain nvcc.

Each .cu is compiled to an object in parallel, then linked into
``libqsa_gb300.so`` next to this file.  Objects are rebuilt when their source,
a shared header or the flags change.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libqsa_gb300.so")
SOURCES = ["api.cu", "block_scores.cu", "topk.cu", "decode_attn.cu", "decode_window.cu", "prompt_attn.cu",
           "noalloc.cu", "kv_append.cu", "tc_rate.cu", "shard.cu", "block_sums.cu"]
HEADERS = [os.path.join(CSRC, h) for h in ("common.cuh", "kernels.h", "tc.cuh", "mma_sync.cuh")] + [
    os.path.join(ROOT, "include", "qsa.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-cudart", "shared",
                "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the QSA CUDA library cannot be built")


def _digest(paths, extra: str) -> str:
    h = hashlib.sha256(extra.encode())
    for p in paths:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _compile(nvcc: str, src: str, verbose: bool) -> str:
    path = os.path.join(CSRC, src)
    tag = _digest([path] + HEADERS, " ".join(FLAGS))
    obj = os.path.join(BUILD, f"{os.path.splitext(src)[0]}-{tag}.o")
    if os.path.exists(obj):
        return obj
    cmd = [nvcc] + FLAGS + ["-c", path, "-o", obj + ".tmp"]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)
    os.replace(obj + ".tmp", obj)
    return obj


def build(verbose: bool = False) -> str:
    """Compile and link the library; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, verbose), SOURCES))
    stamp = os.path.join(BUILD, "lib.stamp")
    key = "|".join(objs)
    if os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == key:
        return LIB
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", LIB + ".tmp"] + objs
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(LIB + ".tmp", LIB)
    with open(stamp, "w") as f:
        f.write(key)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
