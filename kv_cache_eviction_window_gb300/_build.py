"""Build libkvsel.so in-tree with nvcc for sm_103a.

Each CUDA translation unit compiles in parallel to an object under ``_build/``; the
objects link into ``kv_cache_eviction_window_gb300/libkvsel.so`` with the static CUDA
runtime (the TMA tensor-map encoder is looked up through the runtime at first use).
The benchmark's exponential-unit probe (``bench_ex2_probe.cu`` beside ``bench.py``, not
part of the library) builds into its own ``libkvsel_ex2probe.so`` in the same step.
``build()`` is idempotent: it rebuilds when a source or header is newer than its library.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libkvsel.so")
PROBE_SRC = os.path.join(ROOT, "bench_ex2_probe.cu")
PROBE_LIB = os.path.join(ROOT, "libkvsel_ex2probe.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(PROBE_LIB):
        return True
    t = min(os.path.getmtime(LIB), os.path.getmtime(PROBE_LIB))
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    return any(os.path.getmtime(p) > t for p in deps + [PROBE_SRC])


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libkvsel.so; returns its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    def build_probe() -> None:
        tmp = PROBE_LIB + ".tmp"
        cmd = [nvcc, *ARCH, *FLAGS, "-shared", PROBE_SRC, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {PROBE_SRC}:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, PROBE_LIB)

    with ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        probe = ex.submit(build_probe)
        objs = list(ex.map(compile_one, sources()))
        probe.result()
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
