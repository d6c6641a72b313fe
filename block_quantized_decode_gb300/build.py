"""Build libmlq.so (the C-ABI CUDA library) in-tree for sm_103a.

Each .cu file under csrc/ is compiled by nvcc in parallel into _build/,
then linked into block_quantized_decode_gb300/libmlq.so against the shared
CUDA runtime.  No cmake; one -gencode; a minute or less on a few cores.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmlq.so")
# The bounds-checking build (MLQ_CHECK_BOUNDS=1 in the environment, or
# check_bounds=True): every kernel index check records MLQ_E_BOUNDS and skips
# the access; a library of its own so that both builds can coexist.
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libmlq_checked.so")


def check_bounds_requested() -> bool:
    return os.environ.get("MLQ_CHECK_BOUNDS") == "1"
SOURCES = ["capi.cu", "quantize.cu", "matvec.cu", "matvec_tma.cu", "gemm_small_m.cu", "prefetch.cu", "chain.cu", "fused.cu", "gemm_mma.cu", "gemm_mma_cluster.cu", "gemm_umma.cu", "gemm_ring.cu", "phase.cu", "phase_ring.cu", "layer.cu", "stream.cu", "q4k.cu", "nbits.cu", "diag.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmlq")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def up_to_date(lib: str = LIB) -> bool:
    return os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime()


def build(force: bool = False, verbose_ptxas: bool = False, check_bounds: bool | None = None) -> str:
    if check_bounds is None:
        check_bounds = check_bounds_requested()
    lib_out = LIB_CHECKED if check_bounds else LIB
    build_dir = BUILD_CHECKED if check_bounds else BUILD
    if not force and up_to_date(lib_out):
        return lib_out
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                    "-I", CSRC]
    if check_bounds:
        flags.append("-DMLQ_CHECK_BOUNDS")
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [cc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if out and (p.returncode != 0 or verbose_ptxas):
            sys.stderr.write(out.decode(errors="replace"))
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    tmp = lib_out + ".tmp%d" % os.getpid()
    subprocess.run([cc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs, check=True)
    os.replace(tmp, lib_out)
    return lib_out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                check_bounds=True if "--check-bounds" in sys.argv else None))
