"""Build libfdec.so in-tree with nvcc for sm_103a (no cmake, no torch extension machinery).

Each translation unit is compiled in parallel, then linked into one shared
library next to this file.  The CUDA runtime is linked statically (nvcc's
default), so the library only needs the driver at run time; it shares the
device's primary context, streams and events with PyTorch in the same process.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfdec.so")
# Benchmark helper (end-to-end steps timed from C), linked against LIB; not part of the ABI.
E2E_SRC = os.path.join(PKG, "e2e", "e2e_loop.cu")
E2E_LIB = os.path.join(PKG, "libfdec_e2e.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers_mtime() -> float:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hs.append(os.path.join(ROOT, "include", "fdec.h"))
    return max(os.path.getmtime(h) for h in hs)


def build(force: bool = False, verbose: bool = False, jobs: int = 0) -> str:
    """Compile (what changed) and link libfdec.so; returns its path."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    hdr = _headers_mtime()
    srcs = sources()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        if (not force and os.path.exists(obj) and os.path.getmtime(obj) >= os.path.getmtime(src)
                and os.path.getmtime(obj) >= hdr):
            return obj, False
        cmd = [nvcc, *ARCH, *FLAGS, "-c", src, "-o", obj + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        os.replace(obj + ".tmp", obj)
        return obj, True

    n = jobs or min(len(srcs), os.cpu_count() or 4)
    with ThreadPoolExecutor(max_workers=n) as ex:
        results = list(ex.map(compile_one, srcs))
    objs = [o for o, _ in results]
    rebuilt = any(r for _, r in results)
    if rebuilt or force or not os.path.exists(LIB) or any(os.path.getmtime(o) > os.path.getmtime(LIB) for o in objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    _build_e2e(nvcc, force)
    return LIB


def _build_e2e(nvcc: str, force: bool) -> None:
    """libfdec_e2e.so: the C end-to-end loop bench.py times (links libfdec.so via $ORIGIN)."""
    if (not force and os.path.exists(E2E_LIB) and os.path.getmtime(E2E_LIB) >= os.path.getmtime(E2E_SRC)
            and os.path.getmtime(E2E_LIB) >= os.path.getmtime(LIB)):
        return
    tmp = E2E_LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, *FLAGS, "-shared", E2E_SRC, "-o", tmp, "-L", PKG, "-lfdec", "-Xlinker", "-rpath,$ORIGIN"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the e2e helper failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, E2E_LIB)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
