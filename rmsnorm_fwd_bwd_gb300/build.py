"""Build ``librmsnorm.so`` (sm_103a) in-tree with nvcc.

Each ``csrc/*.cu`` file is compiled to an object in parallel, then linked into
one shared library next to this file. Objects and the ptxas resource report go
to ``_build/``. Rebuilds only what is older than its sources.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "librmsnorm.so")
# debug build: the same sources with -DRMSNORM_DEBUG (every TMA read of a row
# kernel is checked against its tensor's extent; see csrc/device.cuh)
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "librmsnorm_debug.so")
HEADER = os.path.join(ROOT, "include", "rmsnorm.h")
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile and link the release library, or with debug=True the debug
    build (librmsnorm_debug.so); returns the library's path."""
    build_dir, lib_path = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    flags = NVCC_FLAGS + (["-DRMSNORM_DEBUG"] if debug else [])
    os.makedirs(build_dir, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))) + HEADERS
    nvcc = _nvcc()
    jobs = []
    for src in sources:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        if force or _stale(obj, [src] + headers):
            jobs.append((src, obj))

    def compile_one(job):
        src, obj = job
        log = obj[:-2] + ".ptxas.txt"
        cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj + ".tmp"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        with open(log, "w") as f:
            f.write(res.stdout + res.stderr)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stderr[-4000:]}")
        os.replace(obj + ".tmp", obj)
        return obj

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            list(ex.map(compile_one, jobs))
    objs = [os.path.join(build_dir, os.path.basename(s)[:-3] + ".o") for s in sources]
    if force or jobs or _stale(lib_path, objs):
        tmp = lib_path + f".{os.getpid()}.tmp"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stderr[-4000:]}")
        os.replace(tmp, lib_path)
    if verbose:
        print(lib_path)
    return lib_path


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv)
