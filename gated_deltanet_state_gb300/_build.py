"""Builds the engine's shared library, libgdn.so, in-tree for sm_103a.

Each CUDA translation unit is compiled by its own nvcc process (in parallel),
the host arithmetic by gcc, and the objects are linked with the static CUDA
runtime.  A stamp of the sources and flags skips the work when nothing changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgdn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-v"]
CU_SOURCES = ["api.cu", "prefill.cu", "replay.cu", "decode.cu", "checkpoint.cu", "noalloc.cu", "tc_replay.cu", "tc_prefill.cu", "tc_chain.cu"]
C_SOURCES = ["gdn_host.c"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the engine needs the CUDA toolkit to build")


def _stamp() -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            with open(os.path.join(d, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    h.update(" ".join(ARCH + NVCC_FLAGS).encode())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libgdn.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    stamp_file = os.path.join(BUILD, "stamp")
    stamp = _stamp()
    if not force and os.path.exists(LIB) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read() == stamp:
                return LIB
    nvcc = _nvcc()
    inc = ["-I", INCLUDE, "-I", CSRC]
    jobs = []
    for src in CU_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        jobs.append(([nvcc, *ARCH, *NVCC_FLAGS, *inc, "-c", os.path.join(CSRC, src), "-o", obj], obj))
    for src in C_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        jobs.append((["gcc", "-O2", "-std=c11", "-fPIC", *inc, "-c", os.path.join(CSRC, src), "-o", obj], obj))

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        logs = list(ex.map(run, [c for c, _ in jobs]))
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        f.write("\n".join(logs))
    if verbose:
        print("\n".join(logs))
    tmp = LIB + f".{os.getpid()}.tmp"
    run([nvcc, *ARCH, "-shared", "-o", tmp, *[o for _, o in jobs]])
    os.replace(tmp, LIB)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
