"""Build libfa.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each .cu file is compiled to an object in parallel, then linked into
``_lib/libfa.so`` next to this file. Re-running only rebuilds when a source
or header is newer than the library. ``build(debug=True)`` builds the
bounds-checked flavour ``_lib/libfa_debug.so`` (-DFA_DEBUG) instead.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libfa.so")
DEBUG_LIB_PATH = os.path.join(OUT_DIR, "libfa_debug.so")
SOURCES = ["fa_api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_noalloc.cu", "fa_softmax.cu", "fa_decode.cu",
           "fa_host.cu", "fa_selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-I", os.path.join(ROOT, "include")]


def _nvcc():
    exe = shutil.which("nvcc")
    if exe is None:
        cand = "/usr/local/cuda/bin/nvcc"
        if os.path.exists(cand):
            return cand
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa.so")
    return exe


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "fa.h"))
    files.append(os.path.abspath(__file__))
    return files


def needs_build(debug: bool = False) -> bool:
    path = DEBUG_LIB_PATH if debug else LIB_PATH
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile and link libfa.so (libfa_debug.so with debug=True); returns
    its path. Raises on failure."""
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    if not force and not needs_build(debug):
        return lib_path
    nvcc = _nvcc()
    build_dir = os.path.join(BUILD_DIR, "debug") if debug else BUILD_DIR
    flavour = ["-DFA_DEBUG"] if debug else []
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(build_dir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *NVCC_FLAGS, *flavour, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
