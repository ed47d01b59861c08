"""Build libtpla.so in-tree with nvcc for sm_103a (B300).

    python -m tensor_column_linear_gelu_b300.build [--force] [--verbose-ptxas] [--checked]

Each csrc/*.cu compiles to an object under _build/, then the objects link into
tensor_column_linear_gelu_b300/libtpla.so against the shared CUDA runtime.
--checked builds libtpla_checked.so instead (objects under _build_checked/):
the same kernels compiled with TPLA_CHECKED, whose index checks record a
failure in the device error word (TP_ERR_DEVICE_CHECK) and skip the access.
The binding loads it when the environment sets TPLA_CHECKED=1.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libtpla.so")
LIB_CHECKED = os.path.join(PKG, "libtpla_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-DNDEBUG",
                     "-Xcompiler", "-fPIC,-O2,-Wall",
                     "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtpla.so")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) +
            glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps() + [__file__])


def build(force: bool = False, verbose_ptxas: bool = False, quiet: bool = True,
          checked: bool = False) -> str:
    lib = LIB_CHECKED if checked else LIB
    bdir = BUILD + "_checked" if checked else BUILD
    if not force and not verbose_ptxas and up_to_date(lib):
        return lib
    nvcc = _nvcc()
    os.makedirs(bdir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if checked:
        extra += ["-DTPLA_CHECKED"]

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, (r.stdout + r.stderr)

    with cf.ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, _sources()))
    if verbose_ptxas or not quiet:
        for obj, log in results:
            if log.strip():
                print(f"== {os.path.basename(obj)}\n{log}", file=sys.stderr)
    tmp = lib + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    ap.add_argument("--checked", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose_ptxas=a.verbose_ptxas, quiet=False, checked=a.checked))
