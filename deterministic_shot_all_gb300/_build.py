"""Builds ``libarx.so`` (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel to an object under ``_build/`` and
nvcc links them into ``deterministic_shot_all_gb300/libarx.so`` with the CUDA
runtime linked statically (the library needs only the driver at run time).

Numerics flags: no fast-math; ``-ftz=false`` keeps fp32 subnormals, which the
bit-exact rank-order sum depends on.

``--bounds-check`` (``build(bounds_check=True)``) builds the checking variant,
``libarx_boundscheck.so``, with ``-DARX_BOUNDS_CHECK``: every data access of the
kernels is checked against its buffer, counted and skipped when outside it.
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
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libarx.so")
CHECK_OBJ_DIR = os.path.join(PKG, "_build_boundscheck")
CHECK_LIB = os.path.join(PKG, "libarx_boundscheck.so")

SOURCES = ["reduce.cu", "step.cu", "abi.cu", "step_noalloc.cu", "external.cu"]
HEADERS = [os.path.join(CSRC, h) for h in ("arx_device.cuh", "arx_internal.h")] + [
    os.path.join(INCLUDE, "arx.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
    "-Xcompiler", "-fPIC,-O2,-Wall", "-I", INCLUDE, "-I", CSRC,
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libarx.so")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, extra: list[str], verbose: bool, obj_dir: str = OBJ_DIR) -> str:
    obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
    path = os.path.join(CSRC, src)
    if _stale(obj, [path, *HEADERS, __file__]) or extra:
        cmd = [nvcc(), *NVCC_FLAGS, *extra, "-c", path, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr, file=sys.stderr)
    return obj


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          bounds_check: bool = False) -> str:
    """Compile (if stale) and return the path of ``libarx.so`` (or of the
    bounds-checking variant)."""
    obj_dir, lib = (CHECK_OBJ_DIR, CHECK_LIB) if bounds_check else (OBJ_DIR, LIB)
    os.makedirs(obj_dir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if bounds_check:
        extra = extra + ["-DARX_BOUNDS_CHECK"]
    if force:
        for s in SOURCES:
            o = os.path.join(obj_dir, os.path.splitext(s)[0] + ".o")
            if os.path.exists(o):
                os.remove(o)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, verbose or ptxas_info, obj_dir), SOURCES))
    if _stale(lib, objs) or force:
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                bounds_check="--bounds-check" in sys.argv))
