"""Builds libqmv.so (the C-ABI library) in-tree with nvcc for sm_103a.

Every .cu unit under csrc/ is compiled in parallel, then linked into
moe_matvec_gb300/_build/libqmv.so.  Rebuilds only when a source is newer than
the library.  build(debug=True) compiles the same sources with QMV_DEBUG (the
kernels' software range checks, see qmv_debug_shrink_outputs in qmv.h) into
moe_matvec_gb300/_build_debug/libqmv_debug.so."""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libqmv.so")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(BUILD_DEBUG, "libqmv_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
          "-I", os.path.join(ROOT, "include")]
# Units whose fp64 arithmetic must not be contracted into FMAs.
NO_FMAD = {"quantize_weights.cu"}


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + [
        os.path.join(ROOT, "include", "qmv.h")]


def up_to_date(debug: bool = False) -> bool:
    lib = LIB_DEBUG if debug else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, debug: bool = False) -> str:
    lib, bdir = (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    if not force and up_to_date(debug):
        return lib
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    flags = COMMON + (["-DQMV_DEBUG"] if debug else [])

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj]
        if os.path.basename(src) in NO_FMAD:
            cmd.insert(1, "-fmad=false")
        if ptxas_info:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for _, err in results:
            if err:
                sys.stderr.write(err)
    tmp = lib + f".{os.getpid()}.tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp] + [o for o, _ in results] + ["-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="-v" in sys.argv, debug="--debug" in sys.argv))
