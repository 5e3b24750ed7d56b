"""Build the CUDA library (libgb300gemm.so) in-tree with nvcc for sm_103a.

Translation units are compiled in parallel (the tcgen05 kernel once per tile
width) and linked into one shared library with the CUDA runtime linked
statically.  The library is rebuilt when a source is newer than it, or when
it does not load on this machine (e.g. it was built for another CPU).
"""
from __future__ import annotations

import concurrent.futures as cf
import ctypes
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libgb300gemm.so")
BUILD_DIR = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         f"-I{INCLUDE}", f"-I{CSRC}"]

# (source, extra defines, object name)
UNITS = [
    ("gemm_host.cu", [], "gemm_host.o"),
    ("aux_kernels.cu", [], "aux_kernels.o"),
    ("noalloc.cu", [], "noalloc.o"),
    ("tc_launch.cu", ["-DTC_BN=256"], "tc_bn256.o"),
    ("tc_launch.cu", ["-DTC_BN=128"], "tc_bn128.o"),
    ("tc_launch.cu", ["-DTC_BN=64"], "tc_bn64.o"),
    ("tc_pair_launch.cu", [], "tc_pair.o"),
    ("decode.cu", [], "decode.o"),
    ("decode_mma.cu", [], "decode_mma.o"),
    ("i8_mma.cu", [], "i8_mma.o"),
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    if any(os.path.getmtime(s) > t for s in _sources()):
        return True
    try:
        ctypes.CDLL(LIB)
    except OSError:
        return True
    return False


def _compile(unit, verbose: bool):
    src, defs, obj = unit
    out = os.path.join(BUILD_DIR, obj)
    cmd = [nvcc(), *ARCH, *FLAGS, *defs, "-c", os.path.join(CSRC, src), "-o", out]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stderr}")
    return out, r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library if needed; return its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        results = list(ex.map(lambda u: _compile(u, verbose), UNITS))
    if verbose:
        for _, log in results:
            if log:
                print(log)
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
