"""Build libnvfp4kv.so (the CUDA kernels + C ABI) in-tree for sm_103a with nvcc.

The translation units compile in parallel; the result lands in ``_build/`` next to this file.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libnvfp4kv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the NVFP4 KV library needs the CUDA toolkit")
    return cand


def _cuda_lib_dir() -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(_nvcc()))), "lib64")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(CSRC, "*.h")) + [os.path.join(ROOT, "include", "nvfp4_kv.h")]


# A second copy of the library whose host code (argument checks, workspace carving, launch
# set-up) is instrumented with AddressSanitizer and UndefinedBehaviorSanitizer, for the host-only
# checks of the C ABI; the device code is the same.
SAN_OUT = os.path.join(OUT, "sanitized")
SAN_LIB = os.path.join(SAN_OUT, "libnvfp4kv.so")
SAN_FLAGS = ["-Xcompiler", "-fsanitize=address", "-Xcompiler", "-fsanitize=undefined",
             "-Xcompiler", "-fno-sanitize-recover=all", "-Xcompiler", "-fno-omit-frame-pointer"]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, sanitize: bool = False) -> str:
    out, lib = (SAN_OUT, SAN_LIB) if sanitize else (OUT, LIB)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(out, exist_ok=True)
    nvcc = _nvcc()
    objs = []
    extra = SAN_FLAGS if sanitize else []

    def compile_one(src):
        obj = os.path.join(out, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(sources())) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".tmp{os.getpid()}"
    # shared CUDA runtime: in a process that already loaded libcudart.so.13 (e.g. through
    # torch) the same instance is reused, so the library and its caller agree on the current
    # device; the rpath lets a plain C caller find the toolkit's copy.
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", *extra, "-o", tmp, *objs,
           "-Xlinker", "-rpath," + _cuda_lib_dir()]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
