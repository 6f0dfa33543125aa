"""Build the CUDA library ``libmoe_gb300.so`` in-tree (sm_103a only).

Each ``csrc/*.cu`` file is compiled in parallel with nvcc into ``_build/``
and linked into ``token_dispatch_grouped_moe_gb300/libmoe_gb300.so``. No
cmake, no torch extension machinery: the library is a plain C-ABI shared
object loaded with ctypes.

    python -m token_dispatch_grouped_moe_gb300.build [--force]
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
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmoe_gb300.so")
SOURCES = ["route.cu", "route_tc.cu", "permute.cu", "permute_static.cu", "grouped_gemm.cu", "combine.cu", "api.cu",
           "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", *ARCH]


def nvcc() -> str:
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: set CUDA_HOME or put nvcc on PATH")


def _deps(src: str) -> list[str]:
    hdrs = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".cuh", ".h"))]
    hdrs.append(os.path.join(ROOT, "include", "moe.h"))
    return [src, *hdrs]


def _stale(out: str, deps: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def _compile(src_name: str, force: bool) -> str:
    src = os.path.join(CSRC, src_name)
    obj = os.path.join(BUILD, src_name.replace(".cu", ".o"))
    if force or _stale(obj, _deps(src)):
        cmd = [nvcc(), *NVCC_FLAGS, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src_name}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, force), SOURCES))
    if force or _stale(LIB, objs):
        tmp = LIB + ".tmp"
        cmd = [nvcc(), "-shared", *ARCH, "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}")
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
