"""Build the C-ABI shared library libzero_gb300.so in-tree for sm_103a.

One nvcc invocation compiles the kernels and the host side and links them
into ``zero_partitioned_mixed_gb300/_build/libzero_gb300.so`` against the
shared CUDA runtime (the same libcudart that PyTorch loads).  Device code is
built with ``-fmad=false`` and IEEE division and square root so every fp32
operation of the step is rounded once, as the method's oracle states it.

Run ``python -m zero_partitioned_mixed_gb300.build`` or call
:func:`build_library`.
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
LIB_NAME = "libzero_gb300.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)

SOURCES = ["zero_kernels.cu", "zero_quant.cu", "zero_tma.cu", "zero_api.cpp", "zero_noalloc.cu"]
HEADERS = [os.path.join(INCLUDE, "zero_gb300.h"), os.path.join(CSRC, "zero_internal.h"),
           os.path.join(CSRC, "zero_device.cuh")]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libzero_gb300.so")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def nvcc_command(out: str = LIB_PATH, extra=None) -> list:
    nvcc = _nvcc()
    cmd = [
        nvcc, ARCH, "-O3", "-lineinfo", "-std=c++17",
        "-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
        "-Xcompiler", "-fPIC,-O2,-ffp-contract=off,-fvisibility=hidden",
        "-Xptxas", "-v",
        "-shared", "-cudart", "shared",
        "-Xlinker", "-rpath," + _cuda_lib_dir(nvcc),
        "-I" + INCLUDE, "-I" + CSRC,
        "-o", out,
    ]
    cmd += [os.path.join(CSRC, s) for s in SOURCES]
    if extra:
        cmd += list(extra)
    return cmd


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile libzero_gb300.so if it is missing or older than its sources."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    # a name of this process's own: several processes (ranks) may build at
    # once; each renames its finished library into place atomically
    tmp = f"{LIB_PATH}.{os.getpid()}.tmp"
    cmd = nvcc_command(out=tmp)
    proc = subprocess.run(cmd, capture_output=True, text=True)
    log = os.path.join(BUILD_DIR, f"build.{os.getpid()}.log")
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n\n" + proc.stdout + proc.stderr)
    if proc.returncode != 0:
        raise RuntimeError("building libzero_gb300.so failed:\n" + proc.stdout + proc.stderr)
    os.replace(tmp, LIB_PATH)
    os.replace(log, os.path.join(BUILD_DIR, "build.log"))
    if verbose:
        sys.stdout.write(proc.stdout + proc.stderr)
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose=True))
