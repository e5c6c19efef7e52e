"""Build libaqpq.so in-tree with nvcc for sm_103a.

Each CUDA translation unit under csrc/ is compiled in parallel to an object
file, then linked into decode_attention_product_gb300/_build/libaqpq.so.
Rebuilds only when a source or header is newer than the library.
"""
from __future__ import annotations

import fcntl
import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libaqpq.so")
# the same sources with AQ_DEBUG_CHECKS: internal invariants reported through
# the device status word (AQ_DEV_INVARIANT); selected by AQPQ_DEBUG_CHECKS=1
DEBUG_BUILD = os.path.join(HERE, "_build_debug")
DEBUG_LIB = os.path.join(DEBUG_BUILD, "libaqpq.so")


def debug_requested() -> bool:
    return os.environ.get("AQPQ_DEBUG_CHECKS") == "1"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libaqpq")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def needs_build(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(d) > t for d in _deps())


def build(force: bool = False, verbose: bool = False, jobs: int | None = None,
          debug: bool | None = None) -> str:
    """Compile and link; returns the library path.  Raises on a compile error.
    `debug` (default: AQPQ_DEBUG_CHECKS=1 in the environment) builds the
    AQ_DEBUG_CHECKS variant into its own directory."""
    if debug is None:
        debug = debug_requested()
    build_dir, lib_path = (DEBUG_BUILD, DEBUG_LIB) if debug else (BUILD, LIB)
    if not force and not needs_build(lib_path):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    # one build at a time per directory (parallel test workers, a child
    # process building while its parent runs): the others wait, then find the
    # library current
    with open(os.path.join(build_dir, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            if not force and not needs_build(lib_path):
                return lib_path
            _compile_and_link(build_dir, lib_path, debug, jobs)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)
    if verbose:
        print("built", lib_path)
    return lib_path


def _compile_and_link(build_dir: str, lib_path: str, debug: bool, jobs: int | None) -> None:
    nvcc = _nvcc()
    srcs = _sources()
    extra = ["-DAQ_DEBUG_CHECKS"] if debug else []

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr[-6000:]}")
        with open(obj + ".ptxas.txt", "w") as f:
            f.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=jobs or min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", *objs, "-o", tmp,
           "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, lib_path)


if __name__ == "__main__":
    build(force=True, verbose=True)
