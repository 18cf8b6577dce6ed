"""Build of the CUDA library libdgemm_gb300.so (sm_103a) with nvcc.

The translation units compile in parallel, then link into one shared
library next to this file (``lib/``).  The build runs wherever the library is
used (the GPU hosts are aarch64, this code is built from source there).

A second variant, libdgemm_gb300_debug.so, is the same sources compiled with
DG_DEBUG=1: device-side bounds, alignment and work-unit checks that record a
failure in the status word and skip the access, and the count-writes mode.
The product library does not contain them.
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
OUT_DIR = os.path.join(PKG, "lib")
OBJ_DIR = os.path.join(PKG, "lib", "obj")
LIB_NAME = "libdgemm_gb300.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)
DEBUG_OBJ_DIR = os.path.join(PKG, "lib", "obj_debug")
DEBUG_LIB_PATH = os.path.join(OUT_DIR, "libdgemm_gb300_debug.so")
# variant -> (library, object folder, extra nvcc flags)
VARIANTS = {"product": (LIB_PATH, OBJ_DIR, []),
            "debug": (DEBUG_LIB_PATH, DEBUG_OBJ_DIR, ["-DDG_DEBUG=1"])}

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libdgemm_gb300.so")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + [os.path.join(INCLUDE, "gemm.h"), os.path.abspath(__file__)])


def up_to_date(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=None,
          variants=("product", "debug")) -> str:
    """Compile and link the library variants whose sources changed (all
    translation units of all variants in one parallel pool); returns the
    product library's path."""
    todo = [v for v in variants if force or not up_to_date(VARIANTS[v][0])]
    if not todo:
        return LIB_PATH
    cc = nvcc()

    def compile_one(job):
        variant, src = job
        _, obj_dir, vflags = VARIANTS[variant]
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [cc] + ARCH + NVCC_FLAGS + vflags + list(extra_flags or []) + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)} ({variant}):\n"
                               f"{r.stderr[-6000:]}")
        if verbose and r.stderr:
            print(r.stderr)
        return variant, obj

    for v in todo:
        os.makedirs(VARIANTS[v][1], exist_ok=True)
    jobs = [(v, src) for v in todo for src in sources()]
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        done = list(ex.map(compile_one, jobs))
    for v in todo:
        path = VARIANTS[v][0]
        objs = [o for vv, o in done if vv == v]
        tmp = path + f".tmp{os.getpid()}"
        r = subprocess.run([cc] + ARCH + ["-shared", "-o", tmp] + objs, capture_output=True,
                           text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed ({v}):\n{r.stderr[-6000:]}")
        os.replace(tmp, path)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
