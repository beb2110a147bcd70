"""Build libtdp.so in-tree: nvcc for sm_103a (one -gencode), g++ for host code.

Translation units compile in parallel, then nvcc links the shared library
(static CUDA runtime).  Rebuilds only when a source or header is newer than
the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtdp.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr"] + ARCH
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall"]


def _nvcc():
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu"))), sorted(glob.glob(os.path.join(CSRC, "*.cpp")))


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build step failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libtdp.so; return its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    cus, cpps = _sources()
    inc = ["-I", INCLUDE, "-I", CSRC]
    jobs = []
    for src in cus:
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
        jobs.append((obj, [nvcc, *NVCC_FLAGS, *inc, "-c", src, "-o", obj]))
    for src in cpps:
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
        jobs.append((obj, ["g++", *CXX_FLAGS, *inc, "-c", src, "-o", obj]))
    with cf.ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
        logs = list(ex.map(lambda j: _run(j[1]), jobs))
    if verbose:
        for log in logs:
            print(log)
    tmp = LIB + f".tmp{os.getpid()}"
    _run([nvcc, "-shared", *ARCH, "-o", tmp, *[j[0] for j in jobs]])
    os.replace(tmp, LIB)
    with open(os.path.join(BUILD_DIR, "ptxas.log"), "w") as fh:
        fh.write("\n".join(logs))
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
