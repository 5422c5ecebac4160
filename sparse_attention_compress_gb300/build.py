"""Build libnsa.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each CUDA source compiles to its own object in parallel, then nvcc links the shared
library with the CUDA runtime linked statically (the driver library is opened at run
time, so loading the library needs no GPU).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libnsa.so")
SOURCES = ["api.cu", "compress.cu", "select.cu", "sparse_fwd.cu", "sparse_bwd.cu", "sparse_bwd_tc.cu", "dense_attn.cu", "dense_tc.cu",
           "decode.cu", "decode_nosa.cu", "noalloc.cu", "nosa.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return exe


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "nsa.h")]
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, extra: list[str], build_dir: str) -> str:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip() and os.environ.get("NSA_BUILD_VERBOSE"):
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, extra: list[str] | None = None, out: str | None = None) -> str:
    """Compile and link libnsa.so (or `out`, with extra nvcc flags); returns its path.
    Skips work when the default library is up to date."""
    extra = list(extra or [])
    lib = out or LIB
    if not force and not extra and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    build_dir = BUILD if not out else os.path.join(BUILD, os.path.basename(out) + ".d")
    os.makedirs(build_dir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, build_dir), SOURCES))
    tmp = lib + f".{os.getpid()}.tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
