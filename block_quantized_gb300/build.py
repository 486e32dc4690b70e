"""Build the CUDA library libgq.so in-tree for sm_103a with nvcc.

Each translation unit compiles in parallel; the objects link into one shared
library with the CUDA runtime linked statically, so the library depends on
nothing but the driver.  Output: block_quantized_gb300/_build/libgq.so.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libgq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
          "--expt-relaxed-constexpr"]
# The codecs must reproduce the reference bit for bit: no FMA contraction.
PER_FILE = {"gq_codec.cu": ["-fmad=false"], "gq_q6k.cu": ["-fmad=false"]}
SOURCES = ["gq_api.cu", "gq_codec.cu", "gq_gemv.cu", "gq_mma.cu", "gq_mma_q0.cu", "gq_skinny.cu", "gq_skinny_q0.cu",
           "gq_kv.cu", "gq_q6k.cu", "gq_q5k.cu"]
HEADERS = ["gq_common.cuh", "gq_internal.h", "gq_mma_sync.cuh", "gq_quant8.cuh", "gq_tc.cuh"]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgq")
    return p


def _newest_input() -> float:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "gq.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def needs_build() -> bool:
    return not os.path.exists(LIB) or os.path.getmtime(LIB) < _newest_input()


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    if not force and not needs_build():
        return LIB
    os.makedirs(OUT, exist_ok=True)
    cc = nvcc()
    extra = list(extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(OUT, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *COMMON, *PER_FILE.get(src, []), *extra, "-c",
               os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None))
