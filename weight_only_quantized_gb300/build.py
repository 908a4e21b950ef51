"""Build the CUDA library in-tree: weight_only_quantized_gb300/lib/libgptq_gb300.so (sm_103a only).

Each translation unit is compiled by its own nvcc process, in parallel, then linked
with the shared CUDA runtime (the same libcudart PyTorch loads, so one runtime
instance serves both).
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "lib")
SO = os.path.join(LIBDIR, "libgptq_gb300.so")
SOURCES = ["api.cu", "repack.cu", "gemm_small.cu", "gemm_small_bf16.cu", "gemm_large.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _newest_input() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "gptq.h"), __file__]
    return max(os.path.getmtime(f) for f in files if os.path.isfile(f))


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if anything changed) and return the path of the shared library."""
    if not force and os.path.exists(SO) and os.path.getmtime(SO) >= _newest_input():
        return SO
    os.makedirs(LIBDIR, exist_ok=True)
    objs = [os.path.join(LIBDIR, os.path.splitext(s)[0] + ".o") for s in SOURCES]

    def compile_one(i: int):
        cmd = [nvcc()] + ARCH + FLAGS + ["-c", os.path.join(CSRC, SOURCES[i]), "-o", objs[i]]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, range(len(SOURCES))))
    for cmd, r in results:
        if verbose or r.returncode:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError(f"nvcc failed for {cmd[-3]}")
    tmp = SO + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        raise RuntimeError("link failed")
    os.replace(tmp, SO)
    return SO


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
