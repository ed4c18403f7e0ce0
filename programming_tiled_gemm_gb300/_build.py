"""Build the CUDA library in-tree: one nvcc process per translation unit, then a link.

Output: ``programming_tiled_gemm_gb300/lib/libgemm_gb300.so`` (sm_103a only), and with
``debug=True`` ``lib/libgemm_gb300_debug.so``: the same sources built with -DGEMM_DEBUG,
whose kernels check every computed global index before the access (see internal.h).
Object files go to ``programming_tiled_gemm_gb300/_build/`` (``_build/debug/``).  Nothing is
installed.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libgemm_gb300.so")
LIB_DEBUG = os.path.join(LIBDIR, "libgemm_gb300_debug.so")

SOURCES = ["api.cu", "ffma.cu", "ffma_tma.cu", "skinny.cu", "skinny_tma.cu", "im2col.cu", "conv_implicit.cu", "conv_tc.cu", "tc_gemm.cu",
           "skinny_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xcompiler", "-Wall"]


def nvcc() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def cuda_lib_dir() -> str:
    root = os.path.dirname(os.path.dirname(os.path.realpath(nvcc())))
    for d in ("lib64", "lib", os.path.join("targets", "sbsa-linux", "lib"), os.path.join("targets", "x86_64-linux", "lib")):
        p = os.path.join(root, d)
        if os.path.isdir(p):
            return p
    return os.path.join(root, "lib64")


def _stale(obj: str, deps: list[str]) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, ptxas_verbose: bool = False, force: bool = False, debug: bool = False) -> str:
    objdir = os.path.join(BUILD, "debug") if debug else BUILD
    lib_path = LIB_DEBUG if debug else LIB
    defines = ["-DGEMM_DEBUG"] if debug else []
    os.makedirs(objdir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "gemm.h"))
    jobs = []
    objs = []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [path] + headers):
            cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *defines, "-I", INCLUDE, "-c", path, "-o", obj]
            if ptxas_verbose:
                cmd += ["-Xptxas", "-v"]
            jobs.append(cmd)

    def run(cmd):
        p = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, p

    failed = []
    with ThreadPoolExecutor(max_workers=min(8, max(1, len(jobs)))) as ex:
        for cmd, p in ex.map(run, jobs):
            if verbose or ptxas_verbose or p.returncode != 0:
                sys.stderr.write(" ".join(cmd) + "\n" + p.stdout + p.stderr)
            if p.returncode != 0:
                failed.append(cmd[-3])
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    if force or jobs or _stale(lib_path, objs):
        tmp = lib_path + ".tmp.%d" % os.getpid()
        libdir = cuda_lib_dir()
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
               "-Xlinker", "-rpath," + libdir, "-L" + libdir]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError("link failed:\n" + p.stdout + p.stderr)
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(verbose=True, ptxas_verbose="-v" in sys.argv, force="-f" in sys.argv, debug="--debug" in sys.argv))
