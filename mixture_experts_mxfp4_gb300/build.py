"""Build the CUDA library (libmoe_mxfp4.so) for sm_103a with nvcc.

Each translation unit compiles in parallel, then one link step makes the shared
library in ``mixture_experts_mxfp4_gb300/_lib``.  The CUDA runtime is linked
statically, so the library loads on a machine without a GPU (for the ABI tests)
and needs only the driver at run time.

build(checked=True) makes the bounds-checked variant, libmoe_mxfp4_checked.so
(compiled with -DMOE_CHECKED=1: every sorted-slot index, route-tile field and
tensor-memory column on the GEMM path is checked before use; a violation sets
bit 9 of the device status word and the access is skipped).  It is a test aid,
the product library is the unchecked one.
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
OUT_DIR = os.path.join(PKG, "_lib")
OBJ_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libmoe_mxfp4.so")
CHECKED_LIB = os.path.join(OUT_DIR, "libmoe_mxfp4_checked.so")
SOURCES = ["api.cu", "route_quant_reduce.cu", "gemm.cu", "gemm_w4a16.cu", "noalloc.cu", "probe.cu"]
HEADERS = ["moe_internal.h", "ptx.cuh", "mx.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _flags(verbose_ptxas: bool, checked: bool = False):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    if checked:
        f += ["-DMOE_CHECKED=1"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, quiet: bool = True,
          checked: bool = False) -> str:
    obj_dir = OBJ_DIR + ("_checked" if checked else "")
    lib = CHECKED_LIB if checked else LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(obj_dir, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "moe_mxfp4.h")]
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(obj_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            cmd = [nvcc(), "-c", s, "-o", o] + _flags(verbose_ptxas, checked)
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        for cmd, r in ex.map(run, jobs):
            if r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
                raise RuntimeError("nvcc failed: " + " ".join(cmd))
            if not quiet or verbose_ptxas:
                sys.stderr.write(r.stdout + r.stderr)
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-Xcompiler", "-fPIC"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, quiet=False,
                checked="--checked" in sys.argv))
