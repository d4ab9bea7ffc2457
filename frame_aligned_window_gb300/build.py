"""Builds libwsattn.so (and the bounds-checking libwsattn_debug.so) in-tree
for sm_103a.

    python frame_aligned_window_gb300/build.py [--force] [--debug]

--debug builds libwsattn_debug.so only: the same sources compiled with
WSATTN_DEBUG, whose kernels check every TMA coordinate, tensor-memory column
range, shared-memory layout, output row and work-item index before the access
and report a failed check through the device status word instead of
faulting (the stand-in for a memory checker in the tests).

(Run by path: importing the package itself requires the built library.)

Each translation unit is compiled by nvcc in parallel (one -gencode, no
cmake), then linked into frame_aligned_window_gb300/libwsattn.so next to this
file.  cudart is linked statically; the driver's tensor-map encoder is looked
up at run time, so the library needs no libcuda at link time.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libwsattn.so")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libwsattn_debug.so")
SOURCES = ["plan.cpp", "prepare.cu", "forward.cu", "api.cu", "prepare_static.cu", "produce.cu"]
HEADERS = ["internal.h", "ptx.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-I", CSRC, "-I", INCLUDE]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(force: bool, lib: str) -> bool:
    if force or not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(INCLUDE, "wsattn.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    lib, bdir = (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    if not _stale(force, lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    flags = NVCC_FLAGS + (["-DWSATTN_DEBUG"] if debug else [])
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(bdir, src.rsplit(".", 1)[0] + ".o")
        objs.append(obj)
        cmd = [nvcc, *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cpp"):
            cmd.insert(1, "-x=cu")
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            failed.append((src, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"), flush=True)
    if failed:
        msg = "\n".join(f"--- {s}\n{o}" for s, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = lib + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    if verbose:
        print(" ".join(link), flush=True)
    subprocess.run(link, check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
