"""Build the sm_103a shared library libdspark.so in-tree with nvcc.

Each CUDA translation unit is compiled in parallel, then linked into
``sample_verify_epilogue_gb300/lib/libdspark.so`` (CUDA runtime linked statically).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libdspark.so")
SOURCES = ("prep.cu", "stream_stats.cu", "finalize.cu", "finalize_warp.cu", "accept.cu", "logprobs.cu", "api.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libdspark.so")


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile every .cu for sm_103a and link libdspark.so; returns the library path."""
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith(".cuh")]
    headers.append(os.path.join(os.path.dirname(PKG), "include", "dspark.h"))
    cc = nvcc()

    def compile_one(src):
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        if force or _stale(o, [s] + headers):
            cmd = [cc, *ARCH, *FLAGS, "-c", s, "-o", o]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
            if verbose:
                print(r.stdout + r.stderr, file=sys.stderr)
        return o

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or _stale(LIB, objs):
        tmp = LIB + ".tmp"
        cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


def build_variant(name: str, defines, sources) -> str:
    """A test build: ``sources`` recompiled with ``defines`` (the other objects shared with
    libdspark.so) and linked into lib/libdspark_<name>.so; returns its path."""
    build()
    vdir = os.path.join(BUILD, name)
    os.makedirs(vdir, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith(".cuh")]
    headers.append(os.path.join(os.path.dirname(PKG), "include", "dspark.h"))
    cc = nvcc()
    objs = []
    for src in SOURCES:
        if src in sources:
            s = os.path.join(CSRC, src)
            o = os.path.join(vdir, src.replace(".cu", ".o"))
            if _stale(o, [s] + headers):
                r = subprocess.run([cc, *ARCH, *FLAGS, *defines, "-c", s, "-o", o], capture_output=True, text=True)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed on {src} ({name}):\n{r.stdout}\n{r.stderr}")
            objs.append(o)
        else:
            objs.append(os.path.join(BUILD, src.replace(".cu", ".o")))
    lib = os.path.join(LIBDIR, f"libdspark_{name}.so")
    if _stale(lib, objs):
        r = subprocess.run([cc, *ARCH, "-shared", "-o", lib + ".tmp", *objs], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed ({name}):\n{r.stdout}\n{r.stderr}")
        os.replace(lib + ".tmp", lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
