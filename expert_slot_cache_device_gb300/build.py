"""Build libftmoe.so (sm_103a) in-tree with nvcc.

Every CUDA translation unit under csrc/ is compiled in parallel for
``-gencode arch=compute_103a,code=sm_103a`` (host C++ units with g++) and linked into
``expert_slot_cache_device_gb300/libftmoe.so`` against the shared CUDA runtime.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libftmoe.so")
LIB_CHECK = os.path.join(PKG, "libftmoe_check.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-cudart", "shared",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC] + ARCH


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


CXX_FLAGS = ["-O3", "-std=c++17", "-fPIC", "-pthread", "-I", INCLUDE]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def cxx() -> str:
    for cand in (os.environ.get("CXX"), shutil.which("g++"), shutil.which("c++")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("no C++ compiler found")


def _deps():
    return sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] + \
        [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]


def up_to_date(lib: str = None) -> bool:
    lib = lib or LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, check: bool = False) -> str:
    """Compile libftmoe.so (or, with check=True, the bounds-checked debug library
    libftmoe_check.so: -DFTMOE_CHECK tests device-side indices before use and records a status
    code instead of touching memory out of bounds; `ftmoe` loads it when FTMOE_CHECKED=1)."""
    lib = LIB_CHECK if check else LIB
    if not force and up_to_date(lib):
        return lib
    bdir = os.path.join(BUILD, "check") if check else BUILD
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DFTMOE_CHECK"] if check else [])

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        if src.endswith(".cpp"):
            cmd = [cxx(), *CXX_FLAGS, *(["-DFTMOE_CHECK"] if check else []), "-c", src, "-o", obj]
        else:
            cmd = [cc, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, "-shared", "-cudart", "shared", *ARCH, "-o", tmp, *objs, "-lpthread", "-ldl",
           "-Xlinker", "-rpath=/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                check="--check" in sys.argv))
