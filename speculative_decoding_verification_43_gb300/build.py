"""Builds libspecverify.so in-tree with nvcc for sm_103a (one -gencode, no cmake), and beside it
libspecverify_debug.so, the same sources with -DSPEC_DEBUG (index-checked kernels, see
include/spec_debug.h).

Every .cu file of both libraries is compiled in parallel, then each set is linked into one shared
library next to this file. The CUDA runtime is linked statically, so the library loads on a
machine without a GPU (the driver is only needed once a CUDA call is made).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libspecverify.so")
DEBUG_LIB_PATH = os.path.join(HERE, "libspecverify_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
         "-Xptxas", "-v" if os.environ.get("SPEC_PTXAS_VERBOSE") else "-O3"]


def nvcc() -> str:
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspecverify.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date() -> bool:
    t = min((os.path.getmtime(p) for p in (LIB_PATH, DEBUG_LIB_PATH) if os.path.exists(p)), default=None)
    if t is None or not (os.path.exists(LIB_PATH) and os.path.exists(DEBUG_LIB_PATH)):
        return False
    return all(os.path.getmtime(d) <= t for d in _deps() + [__file__])


def build(force: bool = False, verbose: bool = False) -> str:
    """Builds both libraries (when a source is newer than either); returns the release path."""
    if not force and up_to_date():
        return LIB_PATH
    cc = nvcc()
    variants = (("release", LIB_PATH, []), ("debug", DEBUG_LIB_PATH, ["-DSPEC_DEBUG"]))
    for name, _, _ in variants:
        os.makedirs(os.path.join(BUILD_DIR, name), exist_ok=True)

    def compile_one(job):
        name, src, extra = job
        obj = os.path.join(BUILD_DIR, name, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src} ({name}):\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    srcs = _sources()
    jobs = [(name, src, extra) for name, _, extra in variants for src in srcs]
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(compile_one, jobs))
    for k, (name, path, _) in enumerate(variants):
        mine = objs[k * len(srcs):(k + 1) * len(srcs)]
        tmp = path + f".tmp{os.getpid()}"
        cmd = [cc, *ARCH, "-shared", "-o", tmp, *mine, "-Xcompiler", "-fPIC"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed ({name}):\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, path)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
