"""Builds the C-ABI CUDA library ``libtpmlp.so`` in-tree for sm_103a with nvcc.

Translation units compile in parallel, then link into one shared library with
the CUDA runtime linked statically (the library only needs the driver at run
time; tensor maps are encoded through the runtime's driver entry point).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libtpmlp.so")
SOURCES = ["tpmlp_api.cu", "gemm_tc.cu", "kernels_misc.cu", "noalloc.cu"]
HEADERS = ["ptx.cuh", "gemm_tc.cuh", "internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtpmlp.so")


def _inputs():
    root = os.path.dirname(PKG)
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(root, "include", "tpmlp.h"))
    return files


def up_to_date(out: str = LIB) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(out: str = LIB, extra_flags=(), force: bool = False, verbose: bool = False) -> str:
    """Compile and link; returns the library path.  extra_flags go to every nvcc call."""
    if not force and not extra_flags and up_to_date(out):
        return out
    nv = nvcc()
    tmpdir = tempfile.mkdtemp(prefix="tpmlp_build_")
    try:
        def compile_one(src):
            obj = os.path.join(tmpdir, os.path.splitext(src)[0] + ".o")
            cmd = [nv, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0 or verbose:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}")
            return obj

        with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
            objs = list(ex.map(compile_one, SOURCES))
        tmp_out = os.path.join(tmpdir, "libtpmlp.so")
        cmd = [nv, *ARCH, "-shared", "-o", tmp_out, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("nvcc link failed")
        os.replace(tmp_out, out) if os.path.dirname(out) == tmpdir else shutil.move(tmp_out, out)
    finally:
        shutil.rmtree(tmpdir, ignore_errors=True)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv))
