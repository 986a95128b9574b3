"""Builds librlk.so in-tree from csrc/*.cu with nvcc for sm_103a only.

Each translation unit compiles in its own nvcc process (in parallel); the
objects are linked into ``_build/librlk.so`` with the CUDA runtime linked
statically. No torch extension machinery is involved: the library is a plain
C ABI (include/rlk.h) loaded through ctypes.

``python -m deterministic_token_logprob_gb300.build [--force] [--verbose-ptxas] [--debug-checks]``

``--debug-checks`` builds the variant with device-side index and tensor-copy coordinate
checks (RLK_DEBUG_CHECKS=1, include/rlk.h) into ``_build_debug/librlk.so``.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "librlk.so")
OUT_DEBUG = os.path.join(PKG, "_build_debug")
DEBUG_LIB = os.path.join(OUT_DEBUG, "librlk.so")

SOURCES = ["rlk_api.cu", "rlk_gemm_fwd.cu", "rlk_gemm_dz.cu", "rlk_gemm_dh.cu", "rlk_gemm_dw.cu", "rlk_gemm_fp8.cu",
           "rlk_quant.cu", "rlk_noalloc.cu"]
HEADERS = [os.path.join(CSRC, f) for f in ("rlk_ptx.cuh", "rlk_gemm.cuh", "rlk_internal.h")] + [
    os.path.join(INCLUDE, "rlk.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--fmad=false", "-Xcompiler", "-fPIC",
         "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources_sha256() -> str:
    """SHA-256 over every source file the library is compiled from (in a fixed order): two
    builds with the same value run the same kernels."""
    h = hashlib.sha256()
    for p in [os.path.join(CSRC, s) for s in SOURCES] + HEADERS:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _stamp(extra) -> str:
    h = hashlib.sha256(sources_sha256().encode())
    h.update(" ".join(ARCH + FLAGS + list(extra)).encode())
    return h.hexdigest()


def build(force: bool = False, verbose_ptxas: bool = False, quiet: bool = True,
          debug_checks: bool = False) -> str:
    """Compile (if sources changed) and return the path of librlk.so (of the debug-checks
    variant with debug_checks=True)."""
    out, lib = (OUT_DEBUG, DEBUG_LIB) if debug_checks else (OUT, LIB)
    os.makedirs(out, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if debug_checks:
        extra = extra + ["-DRLK_DEBUG_CHECKS=1"]
    stamp = _stamp(extra)
    stamp_file = os.path.join(out, "librlk.stamp")
    if not force and os.path.exists(lib) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read().strip() == stamp:
                return lib
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(out, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose_ptxas or not quiet:
        for obj, log in results:
            if log.strip():
                print(f"--- {os.path.basename(obj)}\n{log}", file=sys.stderr)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    ap.add_argument("--debug-checks", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, verbose_ptxas=args.verbose_ptxas, quiet=False,
                debug_checks=args.debug_checks))
