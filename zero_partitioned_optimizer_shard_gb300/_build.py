"""Build the CUDA library libzero_shard.so in-tree (nvcc, sm_103a, parallel compiles)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
OBJ = os.path.join(ROOT, "_build", "zero_shard")
LIB = os.path.join(PKG, "libzero_shard.so")
SOURCES = ["partition.cu", "reduce.cu", "finalize.cu", "adamw.cu", "adamw_variants.cu", "api.cu",
           "noalloc.cu", "fused.cu"]
HEADERS = [os.path.join(CSRC, h) for h in ("zero_internal.h", "adamw_elem.cuh", "reduce_elem.cuh",
                                           "step_scalars.cuh")] + [os.path.join(ROOT, "include", "zero.h")]

ARCH = os.environ.get("ZERO_CUDA_ARCH", "103a")
NVCC_FLAGS = [
    "-O3", "-std=c++17", "-lineinfo",
    f"-gencode=arch=compute_{ARCH},code=sm_{ARCH}",
    # every floating-point operation is the one written: no FMA contraction (explicit
    # __fmaf_rn calls stay fused), IEEE division and square root
    "--fmad=false", "-prec-div=true", "-prec-sqrt=true",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
]


def _stale(out: str, deps: list[str]) -> bool:
    return not os.path.exists(out) or any(os.path.getmtime(out) < os.path.getmtime(d) for d in deps)


def _compile(src: str, extra: list[str]) -> str:
    out = os.path.join(OBJ, os.path.splitext(src)[0] + ".o")
    path = os.path.join(CSRC, src)
    if _stale(out, [path, *HEADERS]):
        subprocess.run(["nvcc", *NVCC_FLAGS, *extra, "-c", path, "-o", out], check=True)
    return out


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    os.makedirs(OBJ, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if force:
        for f in os.listdir(OBJ):
            os.remove(os.path.join(OBJ, f))
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    if force or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.run(["nvcc", "-shared", f"-gencode=arch=compute_{ARCH},code=sm_{ARCH}",
                        "-o", tmp, *objs, "-lcudart"], check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose_ptxas=True))
