"""Build step of the CUDA library: compiles csrc/*.cu for sm_103a (one
translation unit per nvcc process, in parallel) and links libkvq.so in-tree,
next to this file.  Rebuilds only when a source or header is newer than the
shared object."""

from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkvq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvq.so")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(ROOT, "include", "kvq.h"), __file__]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


# The debug build: every kernel checks the index arithmetic it does on the
# device and records KVQ_STATUS_BOUNDS instead of making an access out of
# range (include/kvq.h).  Same sources, its own objects and library.
DEBUG_LIB = os.path.join(BUILD, "debug", "libkvq_debug.so")


def build_debug(force: bool = False) -> str:
    return build(force=force, extra_flags=("-DKVQ_DEBUG_BOUNDS",), lib=DEBUG_LIB,
                 build_dir=os.path.join(BUILD, "debug"))


def build(force: bool = False, verbose: bool = False, extra_flags=(), lib: str = LIB, build_dir: str = BUILD) -> str:
    """Compile and link libkvq.so (or `lib`, from objects in `build_dir`);
    returns its path."""
    if not force and up_to_date(lib):
        return lib
    BUILD_ = build_dir
    os.makedirs(BUILD_, exist_ok=True)
    cc = nvcc()
    inc = ["-I", os.path.join(ROOT, "include")]

    def compile_one(src):
        obj = os.path.join(BUILD_, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *FLAGS, *extra_flags, *inc, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=("-Xptxas", "-v") if "--ptxas-v" in sys.argv else ()))
