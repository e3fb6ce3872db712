"""Build libmoe.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in parallel; the shared library links the CUDA
runtime dynamically so that it shares one runtime with PyTorch.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import platform
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libmoe.so")
# the bounds-checked variant (-DMOE_DEBUG_BOUNDS): its kernels check the
# indices they derive from data and skip out-of-range accesses, flagging them
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(BUILD_DEBUG, "libmoe_debug.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

SOURCES = ["moe_api.cu", "moe_route.cu", "moe_route_tc.cu", "moe_dispatch.cu", "moe_quant.cu", "moe_gemm.cu", "moe_combine.cu",
           "moe_kv.cu", "moe_peak.cu",
           "moe_ffn_decode.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-I" + INCLUDE]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libmoe.so")
    return p


def _key(cc: str, defines=()) -> str:
    """Hash of every source, the header, the flags and the host machine: a
    library built from other sources, with other flags or for another
    machine is rebuilt, whatever the file times say."""
    h = hashlib.sha256()
    files = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)) + [os.path.join(INCLUDE, "moe.h"), __file__]
    for f in files:
        h.update(os.path.basename(f).encode() + b"\0")
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join([cc, *ARCH, *NVCC_FLAGS, *defines, platform.machine()]).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    """Compile libmoe.so (or, with debug_bounds, the bounds-checked
    libmoe_debug.so) unless its stamp matches the sources and flags."""
    out_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug_bounds else (BUILD, LIB)
    defines = ["-DMOE_DEBUG_BOUNDS"] if debug_bounds else []
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    key = _key(cc, defines)
    stamp = lib + ".key"
    if not force and os.path.exists(lib) and os.path.exists(stamp) and open(stamp).read().strip() == key:
        return lib

    def one(src):
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *NVCC_FLAGS, *defines, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {os.path.basename(lib)} failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp, "w") as fh:
        fh.write(key + "\n")
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug_bounds="--debug-bounds" in sys.argv))
