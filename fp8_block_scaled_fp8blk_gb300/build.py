"""Build libfp8blk.so in-tree for GB300 (sm_103a) with nvcc.

Compiles the translation units in ``csrc/`` in parallel and links them into
``_build/libfp8blk.so`` (shared CUDA runtime, so the library shares torch's
runtime and streams).  Rebuilds only when a source or header is newer than the
library.  Usage: ``python -m fp8_block_scaled_fp8blk_gb300.build [--force] [-v]``.
Extra nvcc flags (e.g. ``-lineinfo``-style diagnostics) come from the
``FP8BLK_NVCC_EXTRA`` environment variable; changing them needs ``--force``.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libfp8blk.so")
SOURCES = ["abi.cu", "gemv_e4m3.cu", "gemv_bf16.cu", "gemv_tc.cu", "nvfp4_dequant.cu", "nvfp4_gemv.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libfp8blk")


def _flags(ptxas_verbose: bool) -> list[str]:
    f = ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC,-O2",
         "-I", INCLUDE, "-I", CSRC, *os.environ.get("FP8BLK_NVCC_EXTRA", "").split()]
    if ptxas_verbose:
        f += ["-Xptxas", "-v"]
    return f


def _inputs() -> list[str]:
    return (glob.glob(os.path.join(CSRC, "*")) + [os.path.join(INCLUDE, "fp8blk.h"),
                                                   os.path.abspath(__file__)])


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    if not force and not is_stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    flags = _flags(ptxas_verbose)

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", *ARCH, "-cudart", "shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true", help="print ptxas resource usage")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose, ptxas_verbose=args.verbose))


if __name__ == "__main__":
    main()
