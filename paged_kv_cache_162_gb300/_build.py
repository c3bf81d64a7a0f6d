"""Builds libpagedkv.so in-tree for sm_103a (nvcc, no cmake).

Each translation unit compiles in parallel; the link uses the shared CUDA
runtime so the library and PyTorch share one runtime in a process.

PKV_NVTX=1 in the environment builds the library with an NVTX range around
every C-ABI call (for profilers); the default build has none.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpagedkv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CU_SOURCES = ["runtime.cu", "cache_ops.cu", "decode.cu"]
CXX_SOURCES = ["allocator.cpp", "beam_step.cpp"]


def cuda_home() -> str:
    env = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if env and os.path.exists(os.path.join(env, "bin", "nvcc")):
        return env
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _nvcc() -> str:
    return os.path.join(cuda_home(), "bin", "nvcc")


def _inputs():
    """Every file the library is built from: all of csrc (sources and the
    headers they include), the public header and this script."""
    srcs = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))
            if f.endswith((".cu", ".cuh", ".h", ".cpp"))]
    return srcs + [os.path.join(INCLUDE, "pagedkv.h"), os.path.abspath(__file__)]


FLAGS = os.path.join(BUILD, "flags.txt")


def _defines() -> list[str]:
    return ["-DPKV_NVTX"] if os.environ.get("PKV_NVTX", "") not in ("", "0") else []


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    built = open(FLAGS).read() if os.path.exists(FLAGS) else ""
    if built != " ".join(_defines()):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def _compile(src: str, extra: list[str]) -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    inc = ["-I", INCLUDE, "-I", CSRC]
    if src.endswith(".cu"):
        cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
               "-Xptxas", "-warn-spills", *inc, *extra, "-c", src, "-o", obj]
    else:
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-Wextra", *inc,
               *[x for x in extra if x.startswith("-D")],
               "-I", os.path.join(cuda_home(), "include"), "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    extra = (["-Xptxas", "-v"] if verbose_ptxas else []) + _defines()
    srcs = [os.path.join(CSRC, s) for s in CU_SOURCES + CXX_SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), srcs))
    tmp = LIB + f".tmp{os.getpid()}"
    libdir = os.path.join(cuda_home(), "lib64")
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "shared", *objs, "-o", tmp,
           "-Xlinker", f"-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(FLAGS, "w") as f:
        f.write(" ".join(_defines()))
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
