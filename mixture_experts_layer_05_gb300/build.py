"""Build libgbmoe.so (the CUDA kernels + C ABI) in-tree for sm_103a with nvcc.

Each translation unit compiles in parallel to ``_build/*.o`` at the repository root;
the objects link into ``mixture_experts_layer_05_gb300/libgbmoe.so`` next to this file.
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
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libgbmoe.so")
SOURCES = ["api.cu", "topk.cu", "align.cu", "gemm.cu", "gemm_tn.cu", "gemm_fp8.cu", "fp8.cu", "gemm_fp4.cu", "fp4.cu",
           "combine.cu",
           "align_static.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libgbmoe.so")
    return path


def flags(verbose_ptxas: bool = False) -> list:
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
                "-I", os.path.join(ROOT, "include")]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _compile(src: str, verbose_ptxas: bool, defines=(), build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = ([nvcc()] + flags(verbose_ptxas) + [f"-D{d}" for d in defines]
           + ["-c", os.path.join(CSRC, src), "-o", obj])
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, defines=(), lib: str = LIB,
          build_dir: str = BUILD) -> str:
    """Compile every CUDA source and link libgbmoe.so; returns the library path.

    ``defines`` (NAME=VALUE strings) override compile-time tunables of csrc/kernels.h;
    with ``lib`` / ``build_dir`` such a variant builds next to the default library.
    """
    os.makedirs(build_dir, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    hdrs = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    hdrs.append(os.path.join(ROOT, "include", "gbmoe.h"))
    if (not force and os.path.exists(lib)
            and os.path.getmtime(lib) > max(os.path.getmtime(p) for p in srcs + hdrs)):
        return lib
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, defines, build_dir), SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
