"""In-tree build of libspecverify.so (the CUDA library behind include/spec_verify.h).

nvcc compiles each translation unit for sm_103a only, in parallel, and links a
shared library next to this file. The CUDA runtime is linked shared so that the
library and PyTorch use one runtime instance in a process.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libspecverify.so")
BUILD_DIR = os.path.join(ROOT, "_build")

SOURCES = ["spec_verify.cu", "ngram.cu", "suffix.cu", "metrics.cu", "filter.cu", "candidates.cu",
           "vshard.cu", "cluster.cu", "greedy.cu", "fcommit.cu", "onehot.cu"]
GENCODE = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else (shutil.which("nvcc") or "nvcc")


def _cuda_lib_dir() -> str:
    return os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build_library(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile the CUDA library if needed; returns the .so path."""
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    common = [GENCODE, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              f"-I{INCLUDE}", "--expt-relaxed-constexpr"]
    if ptxas_verbose:
        common += ["-Xptxas", "-v"]
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc, *common, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd))
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    logs = []
    for cmd, p in procs:
        out, _ = p.communicate()
        logs.append(out.decode(errors="replace"))
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed ({' '.join(cmd)}):\n{out.decode(errors='replace')}")
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    link = [nvcc, GENCODE, "-shared", "-cudart", "shared", "-o", tmp, *objs,
            "-Xlinker", f"-rpath,{_cuda_lib_dir()}"]
    if verbose:
        print(" ".join(link))
    subprocess.check_call(link)
    os.replace(tmp, LIB_PATH)
    if verbose or ptxas_verbose:
        print("\n".join(l for l in logs if l.strip()))
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build_library(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))
