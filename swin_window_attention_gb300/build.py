"""Builds libswin_wattn.so in-tree from csrc/*.cu with nvcc for sm_103a.

Each translation unit compiles in its own nvcc process (in parallel), then one link
step produces the shared library next to this file. ``debug=True`` builds the
fault-injection variant libswin_wattn_debug.so from the same sources with
SWIN_WATTN_FAULT_INJECTION defined (include/swin_wattn_debug.h); it is used only by the
tests of the bounded device waits. Run ``python -m swin_window_attention_gb300.build
[--force] [--verbose-ptxas] [--debug]``.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libswin_wattn.so")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libswin_wattn_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build swin_wattn")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def is_stale(debug: bool = False) -> bool:
    lib = LIB_DEBUG if debug else LIB
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(d) > t for d in _deps())


def build(force: bool = False, verbose_ptxas: bool = False, debug: bool = False) -> str:
    lib, bdir = (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    if not force and not is_stale(debug):
        return lib
    nvcc = _nvcc()
    os.makedirs(bdir, exist_ok=True)
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                     "--use_fast_math"]
    if debug:
        common += ["-DSWIN_WATTN_FAULT_INJECTION"]
    if verbose_ptxas:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, "-c", src, "-o", obj] + common
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, _sources()))
    if verbose_ptxas:
        for _, err in results:
            sys.stderr.write(err)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", "-o", tmp] + [o for o, _ in results] + ARCH + [
        "-cudart", "shared", "-Xlinker", "-rpath", "-Xlinker", "/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    ap.add_argument("--debug", action="store_true", help="the fault-injection variant")
    a = ap.parse_args()
    print(build(force=a.force or a.verbose_ptxas, verbose_ptxas=a.verbose_ptxas, debug=a.debug))
