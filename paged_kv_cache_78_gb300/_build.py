"""Build of libpa.so: every CUDA translation unit compiled for sm_103a with
nvcc, in parallel, then linked with the static CUDA runtime.  The build is
skipped when no source or header changed since the last one."""
from __future__ import annotations

import concurrent.futures
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpa.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path:
        return path
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpa.so")


def sources():
    cu = sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))
    hdr = sorted(f for f in os.listdir(CSRC) if f.endswith((".cuh", ".h")))
    return cu, hdr


def _digest(files) -> str:
    h = hashlib.sha256()
    for path in files:
        h.update(path.encode())
        with open(path, "rb") as f:
            h.update(f.read())
    h.update(" ".join(ARCH + CUDA_FLAGS).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False) -> str:
    cu, hdr = sources()
    all_files = [os.path.join(CSRC, f) for f in cu + hdr] + [os.path.join(INCLUDE, "pa.h")]
    digest = _digest(all_files)
    stamp = os.path.join(BUILD, "stamp")
    if not force and os.path.exists(LIB) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return LIB
    os.makedirs(BUILD, exist_ok=True)
    compiler = nvcc()

    def compile_one(name: str) -> str:
        src = os.path.join(CSRC, name)
        obj = os.path.join(BUILD, name + ".o")
        cmd = [compiler] + CUDA_FLAGS + ARCH + ["-c", src, "-o", obj]
        if name.endswith(".cpp"):
            cmd = [compiler, "-x", "c++"] + CUDA_FLAGS + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("compile failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    workers = max(1, min(len(cu), os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        objs = list(ex.map(compile_one, cu))
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [compiler, "-shared"] + ARCH + ["-cudart", "static", "-o", tmp] + objs + \
        ["-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(digest)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
