"""Build libar_gb300.so in-tree: nvcc for the sm_103a kernels, g++ for the host
ABI, compiled in parallel and linked with the static CUDA runtime.

    python -m gradient_sync_gb300.build [--force] [--verbose]
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libar_gb300.so")

CUDA_SOURCES = ["fused.cu", "fused_tma.cu", "step.cu", "pack.cu", "noalloc.cu", "compress.cu"]
CXX_SOURCES = ["api.cpp"]
HEADERS = ["internal.h", "common.cuh", "bulk.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Per-file nvcc flags (none at present).
CUDA_FLAGS: dict = {}


def cuda_home() -> str:
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return cand
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    raise RuntimeError("nvcc not found: set CUDA_HOME")


def _inputs():
    files = [os.path.join(CSRC, f) for f in CUDA_SOURCES + CXX_SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "ar.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"build step failed ({res.returncode}):\n{' '.join(cmd)}\n{res.stdout}{res.stderr}")
    if verbose and (res.stdout or res.stderr):
        print(res.stdout + res.stderr, flush=True)
    return res.stdout + res.stderr


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, defines=(),
          out: str | None = None, build_dir: str | None = None) -> str:
    """Compile every source and link the library. Returns the library path.

    ``defines`` (e.g. ["AR_FUSED_NB=8"]) set the compile-time tuning knobs;
    ``out``/``build_dir`` place a variant build elsewhere."""
    lib = out or LIB
    bdir = build_dir or BUILD
    if not force and out is None and up_to_date():
        return LIB
    cuda = cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    os.makedirs(bdir, exist_ok=True)
    common = ["-O3", "-std=c++17", f"-I{INCLUDE}", f"-I{CSRC}"] + [f"-D{d}" for d in defines]
    jobs = []
    objs = []
    for src in CUDA_SOURCES:
        obj = os.path.join(bdir, src + ".o")
        cmd = [nvcc, *ARCH, "-lineinfo", *common, *CUDA_FLAGS.get(src, []), "-Xcompiler", "-fPIC", "-c",
               os.path.join(CSRC, src), "-o", obj]
        if ptxas_info:
            cmd += ["-Xptxas", "-v"]
        jobs.append(cmd)
        objs.append(obj)
    for src in CXX_SOURCES:
        obj = os.path.join(bdir, src + ".o")
        cmd = ["g++", *common, "-fPIC", "-Wall", f"-I{os.path.join(cuda, 'include')}", "-c",
               os.path.join(CSRC, src), "-o", obj]
        jobs.append(cmd)
        objs.append(obj)
    with ThreadPoolExecutor(len(jobs)) as ex:
        logs = list(ex.map(lambda c: _run(c, verbose), jobs))
    tmp = lib + f".tmp{os.getpid()}"
    _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-Xcompiler", "-fPIC", *objs, "-o", tmp,
          "-lpthread", "-ldl", "-lrt"], verbose)
    os.replace(tmp, lib)
    if ptxas_info:
        print("\n".join(logs))
    return lib


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true")
    a = ap.parse_args(argv)
    print(build(force=a.force, verbose=a.verbose, ptxas_info=a.ptxas_info))


if __name__ == "__main__":
    sys.exit(main())
