"""Builds libpkv.so in-tree with nvcc for sm_103a (no torch headers involved).

    python -m paged_kv_cache_282_gb300.build [--force]

Translation units compile in parallel; the shared library links the CUDA
runtime statically so it loads without a matching libcudart on the path.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_objs")
LIB = os.path.join(HERE, "libpkv.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
SOURCES = ["decode_tc_128.cu", "decode_tc_64.cu", "kernels.cu", "decode_static.cu", "pool.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, "pkv_internal.h"), os.path.join(CSRC, "async_copy.cuh"),
              os.path.join(CSRC, "decode_tc.cuh"), os.path.join(INCLUDE, "pkv.h"), __file__]
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _compile(src: str, extra: list[str], objdir: str) -> str:
    obj = os.path.join(objdir, os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
           "-c", src, "-o", obj, *extra]
    if src.endswith(".cu"):
        cmd += ["-Xptxas", "-warn-spills"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, defines=(), lib: str = LIB, objdir: str = OBJ) -> str:
    """Compiles every source (in parallel) and links `lib`.  `defines` are
    extra preprocessor definitions (name=value strings) for a variant build
    into another `lib` / `objdir`."""
    if not force and not defines and lib == LIB and up_to_date():
        return LIB
    os.makedirs(objdir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    extra += [f"-D{d}" for d in defines]
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, objdir), srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
