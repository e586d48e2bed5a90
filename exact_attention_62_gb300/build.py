"""Builds libattn.so in-tree with nvcc for sm_103a.

Each translation unit under ``csrc/`` is compiled in parallel to an object in
``_build/`` and the objects are linked into ``libattn.so`` next to this file
(the CUDA runtime is linked statically).  A unit is rebuilt only when it or a
header is newer than its object.

``build(bounds_check=True)`` builds the debug variant ``libattn_bounds.so``
(objects in ``_build_bounds/``) with ATTN_BOUNDS_CHECK defined: its kernels
check every global access that is not a TMA copy against its buffer's extent
and report a refused access through attn_check_device_status.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libattn.so")
BUILD_BOUNDS = os.path.join(PKG, "_build_bounds")
LIB_BOUNDS = os.path.join(PKG, "libattn_bounds.so")
INCLUDE = os.path.join(ROOT, "include")
SOURCES = ["api.cu", "fwd_tc.cu", "fwd_f32.cu", "decode.cu", "decode_static.cu", "bwd_tc.cu",
           "fp8.cu", "host_pipeline.cu"]
HEADERS = [os.path.join(CSRC, "ptx.cuh"), os.path.join(CSRC, "common.cuh"), os.path.join(CSRC, "per_device.h"),
           os.path.join(INCLUDE, "attn.h"), os.path.join(INCLUDE, "attn_test.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or install the CUDA toolkit)")


def _flags(verbose_ptxas: bool, bounds_check: bool = False):
    f = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                "--expt-relaxed-constexpr", "-I", INCLUDE]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    if bounds_check:
        f += ["-DATTN_BOUNDS_CHECK"]
    return f


def _stale(src: str, obj: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(p) > t for p in [src] + HEADERS)


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int = 4,
          bounds_check: bool = False) -> str:
    build_dir, lib = (BUILD_BOUNDS, LIB_BOUNDS) if bounds_check else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    objs, todo = [], []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(build_dir, s.replace(".cu", ".o"))
        objs.append(obj)
        if force or verbose_ptxas or _stale(src, obj):
            todo.append((src, obj))

    def compile_one(item):
        src, obj = item
        cmd = [cc] + _flags(verbose_ptxas, bounds_check) + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, r

    failed = []
    with cf.ThreadPoolExecutor(max_workers=max(1, jobs)) as ex:
        for src, r in ex.map(compile_one, todo):
            if r.stdout or r.stderr:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                failed.append(src)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    if todo or not os.path.exists(lib) or any(os.path.getmtime(o) > os.path.getmtime(lib) for o in objs):
        tmp = lib + ".tmp.%d" % os.getpid()
        cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs
        subprocess.check_call(cmd)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="--ptxas-v" in sys.argv,
                bounds_check="--bounds-check" in sys.argv))
