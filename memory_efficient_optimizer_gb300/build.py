"""Builds libmeo_adafactor.so (the C-ABI CUDA library) in-tree with nvcc.

Usage: ``python -m memory_efficient_optimizer_gb300.build [--force]``.
The translation units are compiled in parallel for sm_103a only, then
linked into ``memory_efficient_optimizer_gb300/lib/libmeo_adafactor.so`` with
the CUDA runtime linked statically (the library needs no torch at link time).
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libmeo_adafactor.so")
SOURCES = ["adafactor_kernels.cu", "adafactor_api.cpp", "adafactor_noalloc.cu", "lamb.cu", "came.cu"]
HEADERS = [os.path.join(CSRC, "adafactor_internal.h"), os.path.join(CSRC, "row_panel.cuh"), os.path.join(CSRC, "host_copy.cuh"), os.path.join(INCLUDE, "adafactor.h"),
           os.path.join(INCLUDE, "lamb.h"), os.path.join(INCLUDE, "came.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(LIBDIR, exist_ok=True)
    objdir = os.path.join(LIBDIR, f"_obj{os.getpid()}")
    os.makedirs(objdir, exist_ok=True)
    common = [nvcc(), "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O3",
              "-I" + INCLUDE, "-I" + CSRC] + ARCH
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(objdir, os.path.splitext(src)[0] + ".o")
        cmd = common + ["-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cpp"):
            cmd = common + ["-x", "cu", "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and res.stderr:
            sys.stderr.write(res.stderr)
        return obj

    try:
        with ThreadPoolExecutor(len(SOURCES)) as ex:
            objs = list(ex.map(compile_one, SOURCES))
        tmp = LIB + f".tmp{os.getpid()}"
        res = subprocess.run([nvcc(), "-shared", "-cudart", "static"] + ARCH + objs + ["-o", tmp],
                             capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, LIB)
    finally:
        shutil.rmtree(objdir, ignore_errors=True)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true", help="pass -Xptxas -v")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose))
