"""Compile the CUDA library libflce.so for sm_103a, in-tree.

One translation unit (csrc/flce.cu with its two headers) built with nvcc into
lm_head_loss_gb300/_lib/libflce.so; the CUDA runtime is linked statically and
the driver's tensor-map encoder is looked up at run time, so the library
loads on a machine without a GPU.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import tempfile

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libflce.so")
SOURCES = [os.path.join(CSRC, "flce.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, "tile_gemm.cuh"), os.path.join(CSRC, "tile_gemm_pair.cuh"),
                     os.path.join(CSRC, "ptx_sm103.cuh"),
                     os.path.join(CSRC, "vocab_sort.cuh"),
                     os.path.join(INCLUDE, "flce.h")]
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libflce.so")


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(p) <= t for p in DEPENDS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Build libflce.so if it is missing or older than its sources; return its path."""
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(LIB_DIR, exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=LIB_DIR)
    os.close(fd)
    cmd = [nvcc_path(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xptxas", "-v",
           "-shared", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-o", tmp, *SOURCES]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        os.unlink(tmp)
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    if verbose:
        print(res.stdout + res.stderr)
    with open(os.path.join(LIB_DIR, "ptxas_info.txt"), "w") as f:
        f.write(res.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
