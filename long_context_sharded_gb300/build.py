"""Build libmercury_attn.so in-tree with nvcc for sm_103a (GB300).

Each .cu file compiles in parallel to an object; the objects link into one
shared library with the CUDA runtime linked statically, so loading it needs no
libcudart on the library path.  The tensor-map encoder is taken from the
driver at run time (cudaGetDriverEntryPointByVersion), so there is no link-time
dependency on libcuda either.

build(check=True) makes the checked variant in _lib_check/: the same sources
compiled with -DMERCURY_CHECK, whose kernels test every TMA coordinate and
output index before using it and report a bad one as MERCURY_EBOUNDS instead
of touching memory (a debugging build; the binding loads it when the
environment sets MERCURY_CHECKED_BUILD=1).
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB_DIR = os.path.join(HERE, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libmercury_attn.so")
CHECK_LIB_DIR = os.path.join(HERE, "_lib_check")
CHECK_LIB_PATH = os.path.join(CHECK_LIB_DIR, "libmercury_attn.so")
SOURCES = ["api.cu", "attn_fwd.cu", "lse_merge.cu", "noalloc.cu", "gemm_shifted.cu", "schedule.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmercury_attn.so")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(HERE, "..", "include", "mercury_attn.h"))
    return files


def up_to_date(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, check: bool = False) -> str:
    lib_dir, lib_path = (CHECK_LIB_DIR, CHECK_LIB_PATH) if check else (LIB_DIR, LIB_PATH)
    if not force and up_to_date(lib_path):
        return lib_path
    nvcc = _nvcc()
    obj_dir = os.path.join(lib_dir, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    defines = ["-DMERCURY_CHECK"] if check else []

    def compile_one(src):
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *defines, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + ".tmp%d" % os.getpid()
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force=True, verbose=True))
