"""Build the CUDA library (libtq.so) in-tree for sm_103a.

Compiles each translation unit in parallel (nvcc for the kernels, the host C++
through nvcc too) and links one shared library with the CUDA runtime linked
statically, so the library does not depend on which libcudart the process
loaded first.  Usage: ``python -m rotated_quantized_kv_gb300.build``.
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
OBJ = os.path.join(ROOT, "_build", "obj")
LIB = os.path.join(PKG, "_lib", "libtq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_SOURCES = ["tq_compress.cu", "tq_compress_dense.cu", "tq_decode.cu", "tq_mass.cu", "tq_static.cu",
                "tq_generic.cu", "tq_compress_rows.cu", "tq_compress_rows_nh2.cu", "tq_compress_rows_nh4.cu",
                "tq_compress_rows_np2.cu"] + [
                f"tq_decode_kb{k}.cu" for k in range(1, 9)] + [
                f"tq_decode_wide_kb{k}.cu" for k in range(1, 9)]
HOST_SOURCES = ["tq_host.cpp"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtq.so")


def _sources():
    return [os.path.join(CSRC, s) for s in CUDA_SOURCES + HOST_SOURCES] + [
        os.path.join(CSRC, h) for h in ("tq_internal.h", "tq_decode_common.cuh", "tq_decode_packed.cuh",
                                        "tq_mass.h", "tq_decode_geometry.h", "tq_compress_rows.cuh")] + [
        os.path.join(ROOT, "include", "tq.h")]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in _sources())


def _compile(src: str, verbose: bool) -> str:
    out = os.path.join(OBJ, os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
           f"-I{os.path.join(ROOT, 'include')}", "-c", src, "-o", out]
    if verbose and src.endswith(".cu"):
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose:
        sys.stderr.write(r.stderr)
    return out


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libtq.so if any source is newer than it; return its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(OBJ, exist_ok=True)
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in CUDA_SOURCES + HOST_SOURCES]
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), srcs))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
