"""Build libm4q.so in-tree: one nvcc per translation unit (in parallel), for
sm_103a only, then one shared-library link against the shared CUDA runtime.
--bounds builds the bounds-checked variant (-DM4Q_BOUNDS=1, every computed
access tested before it is made) as libm4q_bounds.so beside it.

    python -m swiglu_block_quantized_gb300.buildlib [--force] [--debug] [--bounds]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libm4q.so")
LIB_BOUNDS = os.path.join(OUT_DIR, "libm4q_bounds.so")
SOURCES = ["api.cu", "misc.cu", "gemv.cu", "tc_q4_0.cu", "tc_q8_0.cu", "tc_q2_0.cu", "tc_mlx4.cu", "noalloc.cu", "attention.cu", "attention_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
        os.path.join(os.path.dirname(HERE), "include", "m4q.h"), os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, debug: bool = False, verbose: bool = False, bounds: bool = False) -> str:
    lib = LIB_BOUNDS if bounds else LIB
    if not force and up_to_date(lib):
        return lib
    out_dir = os.path.join(OUT_DIR, "bounds") if bounds else OUT_DIR
    os.makedirs(out_dir, exist_ok=True)
    flags = ["-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall"]
    flags += ["-O0", "-G"] if debug else ["-O3"]
    if bounds:
        flags += ["-DM4Q_BOUNDS=1"]
    if verbose:
        flags += ["-Xptxas", "-v"]
    objs = []

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc(), *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--debug", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--bounds", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, debug=a.debug, verbose=a.verbose, bounds=a.bounds))
