"""Build the native library (``_build/liblp.so``) with nvcc for sm_103a only.

``csrc/lp_api.cu`` holds the handle-based C ABI and ``csrc/lp_noalloc.cu`` the
no-allocation entry point; both instantiate the same kernel templates from
``csrc/kernels.cuh`` with the same flags, so they share the pinned numerics.  The library links
only the shared CUDA runtime (every kernel, the backward's GEMMs included, is its own) and
resolves the driver's tensor-map encoder at run time (no link against libcuda).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liblp.so")
SOURCES = [os.path.join(CSRC, "lp_api.cu"), os.path.join(CSRC, "lp_noalloc.cu"),
           os.path.join(CSRC, "lp_contract.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("kernels.cuh", "numerics.cuh", "ptx.cuh",
                                                  "rl_kernels.cuh", "lp_internal.h",
                                                  "fp8_kernels.cuh", "grad_gemm.cuh")] + [
    os.path.join(INCLUDE, "lp.h")]

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", *ARCH_FLAGS, "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-shared", "-cudart", "shared",
              "-I", INCLUDE, "-I", CSRC]
LINK_FLAGS: list = []


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build liblp.so")
    return path


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile liblp.so if it is missing or older than its sources; return its path."""
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, *(["-Xptxas", "-v"] if verbose else []), "-o", tmp, *SOURCES, *LINK_FLAGS]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + proc.stdout + proc.stderr)
    if verbose:
        sys.stderr.write(proc.stdout + proc.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
