"""In-tree build of libhwkv.so for sm_103a with nvcc (no torch extension machinery).

The translation units compile in parallel, then link into
``head_budgeted_kv_gb300/_build/libhwkv.so`` with the CUDA runtime linked statically.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libhwkv.so")

SOURCES = ("hwkv_host.cpp", "hwkv_copy.cu", "hwkv_decode_simt.cu", "hwkv_decode_tc.cu", "hwkv_noalloc.cu", "hwkv_prefill.cu")
HEADERS = (os.path.join(CSRC, "hwkv_internal.h"), os.path.join(CSRC, "hwkv_device.cuh"),
           os.path.join(CSRC, "hwkv_tcgen05.cuh"), os.path.join(CSRC, "hwkv_decode_tile.cuh"),
           os.path.join(INCLUDE, "hwkv.h"))
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libhwkv.so")
    return path


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, extra) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    path = os.path.join(CSRC, src)
    if _stale(obj, (path,) + HEADERS):
        cmd = [nvcc(), "-c", *ARCH, *FLAGS, *extra, "-o", obj, path]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    return obj


def build(force: bool = False, extra_flags=()) -> str:
    """Compile and link libhwkv.so if any source or header is newer than it."""
    os.makedirs(BUILD, exist_ok=True)
    if force:
        for f in os.listdir(BUILD):
            os.remove(os.path.join(BUILD, f))
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, list(extra_flags)), SOURCES))
    if _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc(), "-shared", *ARCH, "-o", tmp, *objs]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link of libhwkv.so failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build())
