"""Build ``libxfa.so`` in-tree from ``csrc/`` for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library under ``bwd_xfa_fwd_gb300/_build/``.  Only the sm_103a target
is generated (``-gencode arch=compute_103a,code=sm_103a``).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libxfa.so")
SOURCES = ("xfa_api.cu", "aux.cu", "simt.cu", "tc_fwd.cu", "tc_bwd.cu", "tc_dq.cu", "tf_fwd.cu", "tf_bwd.cu", "noalloc.cu", "keep.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _cuda_lib_dir() -> str:
    return os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64")


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every CUDA source and link ``_build/libxfa.so``; returns its path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "xfa.h"))
    nvcc = _nvcc()
    common = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-I", INCLUDE, "-I", CSRC, "-Xcompiler", "-fPIC",
                     "-Xptxas", "-v" if verbose else "-O3"]

    def compile_one(src):
        obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + ".o")
        path = os.path.join(CSRC, src)
        if force or _stale(obj, [path] + headers):
            tmp = obj + f".tmp{os.getpid()}"
            r = subprocess.run([nvcc] + common + ["-c", path, "-o", tmp], capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
            os.replace(tmp, obj)
            if verbose:
                print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs + [
            "-Xlinker", "-rpath," + _cuda_lib_dir()]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
