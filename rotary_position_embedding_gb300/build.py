"""Builds librope_gb300.so in-tree with nvcc for sm_103a.

The four translation units compile in parallel (``nvcc -c``) and link into
one shared library with the CUDA runtime linked statically, so the library
loads on a machine without a GPU driver (every entry point then fails with
ROPE_ERR_CUDA once it reaches a CUDA call; argument checks still run).
"""

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_lib")
LIB_PATH = os.path.join(OUT_DIR, "librope_gb300.so")
SOURCES = ["rope_api.cu", "k_rope.cu", "k_mrope.cu", "k_fused.cu", "k_tma.cu", "k_qkv.cu", "k_mrope_qkv.cu", "k_qkv_tma.cu", "k_mrope_qkv_tma.cu",
           "k_mrope_heads.cu", "k_qkv_heads.cu", "no_alloc.cu"]
HEADERS = ["rope_kernels.cuh", "rope_internal.h", "rope_tma.cuh", "rope_qkv.cuh", "rope_qkv_tma.cuh", "rope_packed.cuh", "rope_fused.cuh",
           "rope_mrope_heads.cuh", "rope_qkv_heads.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librope_gb300.so")


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "rope.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(path=LIB_PATH):
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build_library(force=False, extra_flags=(), out_path=None, verbose=False):
    """Compile (if needed) and return the path of the shared library."""
    out_path = out_path or LIB_PATH
    if not force and not extra_flags and up_to_date(out_path):
        return out_path
    nvcc = nvcc_path()
    obj_dir = os.path.join(os.path.dirname(out_path), f"_obj{os.getpid()}")
    os.makedirs(obj_dir, exist_ok=True)
    common = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "-I", INCLUDE, "-I", CSRC, *extra_flags]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
        cmd = common + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out_path)
    shutil.rmtree(obj_dir, ignore_errors=True)
    return out_path


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))
