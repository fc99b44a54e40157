"""Builds the in-tree shared library libfa_gb300.so for sm_103a with nvcc.

Each translation unit compiles in its own nvcc process (in parallel) and the objects
link into one shared library next to this file.  A stamp of the source hashes and
flags skips the rebuild when nothing changed.  No cmake, one -gencode.
"""

from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libfa_gb300.so")
SOURCES = ["fa_api.cu", "fa_bwd_main.cu", "fa_bwd_split.cu", "fa_bwd_aux.cu", "fa_fwd_tc.cu",
           "fa_wide.cu", "fa_noalloc.cu"]
HEADERS = ["fa_ptx.cuh", "fa_kernels.h", "fa_tiles.h", "fa_bwd_common.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libfa_gb300.so")


def _stamp(extra_flags) -> str:
    h = hashlib.sha256()
    for f in SOURCES + HEADERS:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    with open(os.path.join(ROOT, "include", "fa.h"), "rb") as fh:
        h.update(fh.read())
    h.update(" ".join(ARCH + FLAGS + list(extra_flags)).encode())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def build(verbose: bool = False, extra_flags=(), force: bool = False, lib_path: str = LIB,
          tag: str = "") -> str:
    """Compile and link; `lib_path` / `tag` give variant builds (e.g. with -DFA_TRACE)
    their own library file and object directory."""
    build_dir = os.path.join(BUILD, tag) if tag else BUILD
    os.makedirs(build_dir, exist_ok=True)
    stamp_path = os.path.join(build_dir, "libfa_gb300.stamp")
    stamp = _stamp(extra_flags)
    if not force and os.path.exists(lib_path) and os.path.exists(stamp_path):
        with open(stamp_path) as fh:
            if fh.read() == stamp:
                return lib_path
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr, flush=True)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp_path, "w") as fh:
        fh.write(stamp)
    return lib_path


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
