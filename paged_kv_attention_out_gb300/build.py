"""Builds the pkv CUDA library (libpkv.so) in-tree with nvcc for sm_103a.

Each .cu file under csrc/ compiles to an object in parallel; the objects
link into one shared library that exports the C ABI of include/pkv.h and
uses the shared CUDA runtime (the one PyTorch also loads).
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libpkv.so")
SOURCES = ["pkv_api.cu", "kv_store.cu", "decode.cu", "extend.cu", "cascade.cu", "merge.cu",
           "decode_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the pkv library cannot be built")


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "pkv.h"))
    files.append(os.path.abspath(__file__))
    return files


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def flags(extra=()) -> list[str]:
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC, *extra]


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Compile csrc/*.cu and link libpkv.so; returns the library path."""
    if not force and not is_stale():
        return LIB
    os.makedirs(os.path.join(BUILD, "obj"), exist_ok=True)
    cc = nvcc()
    tag = f"{os.getpid()}"

    def compile_one(src):
        obj = os.path.join(BUILD, "obj", src.replace(".cu", f".{tag}.o"))
        cmd = [cc, *flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".{tag}.tmp"
    # -z defs: a declared but undefined function fails the link here instead
    # of failing to load (or to resolve) at run time
    cmd = [cc, *ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-z", "-Xlinker", "defs",
           "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    for o in objs:
        os.remove(o)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
