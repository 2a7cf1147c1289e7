"""Build libdspark.so (sm_103a) in place with nvcc.

Each translation unit is compiled in parallel, then linked into one shared
library next to this file.  The only target is sm_103a; the build needs no GPU.
build(bounds=True) makes the bounds-checked variant, libdspark_bounds.so, compiled
with -DDSPARK_BOUNDS: every index the kernels compute from data before an access is
checked against its buffer (DSPARK_ERR_BOUNDS, the access sent to element 0).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdspark.so")
BUILD_BOUNDS = os.path.join(HERE, "_build_bounds")
LIB_BOUNDS = os.path.join(HERE, "libdspark_bounds.so")
SOURCES = ["api.cu", "schedule.cu", "schedule_noalloc.cu", "verify.cu", "draft_simt.cu", "draft_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                   "--expt-relaxed-constexpr", *extra]


def _newest_input() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "dspark.h"), __file__]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, bounds: bool = False) -> str:
    lib, bdir = (LIB_BOUNDS, BUILD_BOUNDS) if bounds else (LIB, BUILD)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input():
        return lib
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DDSPARK_BOUNDS"] if bounds else [])

    def compile_one(src):
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        cmd = [cc, *_flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, err in results:
            if err:
                sys.stderr.write(err)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                bounds="--bounds" in sys.argv))
