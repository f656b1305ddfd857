"""Build libfa.so (the CUDA kernels and the C ABI) in-tree with nvcc, for sm_103a.

Each translation unit compiles in its own nvcc process, in parallel, into
``_build/``; the objects are then linked into ``exact_attention_29_gb300/libfa.so``.
Run ``python -m exact_attention_29_gb300.build`` or call ``build()``.

``build(debug=True)`` (``--debug``) makes ``libfa_debug.so`` instead, compiled
with FA_DEBUG: at the end of each pipelined kernel the roles' protocol counts
(items, ring positions, barrier phases, tiles) are compared, and a mismatch is
reported by fa_check_device_error as FA_ERR_CHECK. The binding loads it when
FA_LIBRARY names it.
"""
from __future__ import annotations

import concurrent.futures as cf
import contextlib
import fcntl
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa.so")
DEBUG_OUT_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB = os.path.join(PKG, "libfa_debug.so")
SOURCES = ["fa_api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_decode.cu", "fa_decode_gqa.cu", "fa_quant.cu", "fa_selftest.cu", "fa_noalloc.cu"]
HEADERS = ["sm103.cuh", "fa_common.cuh", "fa_mma.cuh", "fa_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                     "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    paths.append(os.path.join(os.path.dirname(PKG), "include", "fa.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


@contextlib.contextmanager
def _exclusive(path: str):
    """Serialise builds: several processes (one per rank) may call build() at once."""
    with open(path, "w") as f:
        fcntl.flock(f, fcntl.LOCK_EX)
        try:
            yield
        finally:
            fcntl.flock(f, fcntl.LOCK_UN)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, debug: bool = False) -> str:
    """Compile every translation unit and link libfa.so (libfa_debug.so with
    debug=True); returns its path."""
    lib_path, out_dir = (DEBUG_LIB, DEBUG_OUT_DIR) if debug else (LIB, OUT_DIR)
    if not force and os.path.exists(lib_path) and os.path.getmtime(lib_path) >= _newest_input():
        return lib_path
    os.makedirs(out_dir, exist_ok=True)
    with _exclusive(os.path.join(out_dir, ".build.lock")):
        # another process may have built it while this one waited
        if not force and os.path.exists(lib_path) and os.path.getmtime(lib_path) >= _newest_input():
            return lib_path
        return _build_locked(lib_path, out_dir, verbose, ptxas_info, debug)


def _build_locked(lib_path: str, out_dir: str, verbose: bool, ptxas_info: bool, debug: bool) -> str:
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if debug:
        extra = extra + ["-DFA_DEBUG"]

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [nvcc] + NVCC_FLAGS + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                debug="--debug" in sys.argv))
