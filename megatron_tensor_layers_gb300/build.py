"""Build the in-tree CUDA library ``libtp_gb300.so`` for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled by nvcc in parallel, then
linked into one shared library with the CUDA runtime linked statically (the
library's only external dependency is the NVIDIA driver, loaded at run
time).  ``build()`` skips the work when the library is newer than every
source and header.
"""

from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libtp_gb300.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH_FLAGS + [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
    "-I", INCLUDE, "-I", CSRC, "-Xptxas", "-v",
]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libtp_gb300.so")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    lib_m = os.path.getmtime(LIB_PATH)
    deps = _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]
    return all(os.path.getmtime(d) <= lib_m for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library; returns its path."""
    if not force and _up_to_date():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    procs = []
    objs = []
    for src in _sources():
        obj = os.path.join(BUILD_DIR, os.path.basename(src).replace(".cu", ".o"))
        log = obj + ".log"
        objs.append(obj)
        cmd = [nvcc] + NVCC_FLAGS + ["-c", src, "-o", obj]
        procs.append((cmd, log, subprocess.Popen(cmd, stdout=open(log, "w"), stderr=subprocess.STDOUT)))
    failed = []
    for cmd, log, p in procs:
        if p.wait() != 0:
            failed.append((cmd, log))
    if failed:
        msgs = []
        for cmd, log in failed:
            with open(log) as f:
                msgs.append(" ".join(cmd) + "\n" + f.read()[-6000:])
        raise RuntimeError("nvcc failed:\n" + "\n\n".join(msgs))
    tmp = LIB_PATH + ".tmp"
    link = [nvcc] + ARCH_FLAGS + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + " ".join(link) + "\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB_PATH)
    if verbose:
        for obj in objs:
            with open(obj + ".log") as f:
                sys.stdout.write(f.read())
    return LIB_PATH


ABI_OVERHEAD_SRC = os.path.join(PKG, "abi_overhead", "abi_overhead.c")
ABI_OVERHEAD_BIN = os.path.join(BUILD_DIR, "abi_overhead")


def build_abi_overhead() -> str:
    """Compile the host-overhead probe (a C program that times enqueues of
    the C-ABI entry points with no Python in the loop) against the library;
    returns the executable's path."""
    lib = build()
    if os.path.exists(ABI_OVERHEAD_BIN) and os.path.getmtime(ABI_OVERHEAD_BIN) >= max(
            os.path.getmtime(lib), os.path.getmtime(ABI_OVERHEAD_SRC)):
        return ABI_OVERHEAD_BIN
    cuda = os.path.dirname(os.path.dirname(_nvcc()))
    os.makedirs(BUILD_DIR, exist_ok=True)
    cmd = [shutil.which("gcc") or "gcc", "-O2", "-I", INCLUDE, "-I", os.path.join(cuda, "include"), ABI_OVERHEAD_SRC,
           "-L", PKG, "-ltp_gb300", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           "-Wl,-rpath," + PKG + ":" + os.path.join(cuda, "lib64"), "-o", ABI_OVERHEAD_BIN]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("gcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return ABI_OVERHEAD_BIN


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
