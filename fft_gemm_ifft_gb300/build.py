"""Build the CUDA library ``libfno.so`` in-tree for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled by nvcc in parallel, then
linked into ``fft_gemm_ifft_gb300/libfno.so`` (git-ignored).  The build is
skipped when the library is newer than every source and header.
``build(debug_bounds=True)`` makes the index-checking variant
``libfno_bounds.so`` (compiled with FNO_DEBUG_BOUNDS: a global-memory index
out of range records FNO_ERR_DEVICE_BOUNDS and the access is skipped); the
binding loads it instead when FNO_LIBRARY=bounds is set.  Set
``FNO_PTXAS_VERBOSE=1`` to print the register / shared-memory report of each
kernel, and ``FNO_EXTRA_NVCC_FLAGS`` to pass tuning macros (e.g. ``-DFNO_TARGET_GROUPS=4``).
"""
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
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libfno.so")
BOUNDS_BUILD_DIR = os.path.join(HERE, "_build_bounds")
BOUNDS_LIB_PATH = os.path.join(HERE, "libfno_bounds.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfno.so")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def _flags():
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
    if os.environ.get("FNO_PTXAS_VERBOSE"):
        f += ["-Xptxas", "-v"]
    extra = os.environ.get("FNO_EXTRA_NVCC_FLAGS")
    if extra:
        f += extra.split()
    return f


def up_to_date(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    lib_path = BOUNDS_LIB_PATH if debug_bounds else LIB_PATH
    build_dir = BOUNDS_BUILD_DIR if debug_bounds else BUILD_DIR
    if not force and up_to_date(lib_path):
        return lib_path
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    flags = _flags() + (["-DFNO_DEBUG_BOUNDS"] if debug_bounds else [])
    objs = []

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        if verbose or os.environ.get("FNO_PTXAS_VERBOSE"):
            sys.stderr.write(r.stderr)
        return obj

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                debug_bounds="--debug-bounds" in sys.argv))
