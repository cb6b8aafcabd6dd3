"""Builds libstrata_moe.so in-tree with nvcc for sm_103a (GB300).

Each .cu file compiles to an object in parallel, then one shared library is
linked next to this file.  A stamp of the sources' contents and the flags
skips rebuilding when nothing changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libstrata_moe.so")
# the same library with the persistent kernel's phase timestamps recorded
# (STRATA_PX_TRACE): a separate file, never the one the package loads
TRACE_BUILD_DIR = os.path.join(HERE, "_build_trace")
TRACE_LIB_PATH = os.path.join(HERE, "libstrata_moe_trace.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libstrata_moe")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stamp(flags) -> str:
    h = hashlib.sha256()
    files = _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        sorted(glob.glob(os.path.join(CSRC, "*.h"))) + [os.path.join(INCLUDE, "strata_moe.h")]
    for f in files:
        h.update(f.encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(flags).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, trace: bool = False) -> str:
    """The library (trace: the phase-traced one at TRACE_LIB_PATH); returns its path."""
    build_dir, lib_path = (TRACE_BUILD_DIR, TRACE_LIB_PATH) if trace else (BUILD_DIR, LIB_PATH)
    flags = NVCC_FLAGS + (["-DSTRATA_PX_TRACE=1"] if trace else [])
    os.makedirs(build_dir, exist_ok=True)
    stamp_file = os.path.join(build_dir, "stamp")
    stamp = _stamp(flags)
    if not force and os.path.exists(lib_path) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read() == stamp:
                return lib_path
    cc = nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *flags, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib_path + f".{os.getpid()}.tmp"
    r = subprocess.run([cc, *ARCH, "-shared", "--cudart", "static", "-o", tmp, *objs],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return lib_path


if __name__ == "__main__":
    print(build(force=True, verbose=True))
