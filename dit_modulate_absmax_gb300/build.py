"""Builds libh3fp4.so (the C-ABI library) in-tree for sm_103a with nvcc.

Steps: generate the silu table include, compile each .cu translation unit in
parallel (-gencode arch=compute_103a,code=sm_103a, no fast-math), link a
shared library next to this file.  Rebuilds only when a source is newer than
the library.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libh3fp4.so")
SOURCES = ["api.cu", "producer.cu", "gemm.cu", "noalloc.cu"]
HEADERS = ["ptx.cuh", "launch.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else "nvcc")
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC, "-I", BUILD]


def _newest(paths):
    return max(os.path.getmtime(p) for p in paths)


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS + ["gen_silu_lut.py"]]
    files.append(os.path.join(INCLUDE, "h3fp4.h"))
    files.append(os.path.abspath(__file__))
    return files


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest(_inputs()):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    lut = os.path.join(BUILD, "silu_lut.inc")
    gen = os.path.join(CSRC, "gen_silu_lut.py")
    if force or not os.path.exists(lut) or os.path.getmtime(lut) < os.path.getmtime(gen):
        subprocess.check_call([sys.executable, gen, lut])

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [NVCC, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-lcudart_static", "-ldl", "-lpthread", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
