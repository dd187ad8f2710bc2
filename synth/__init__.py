"""Seeded synthetic inputs for the ZeRO optimizer step (host and device twins).

Generates gradient replicas and optimizer state from a counter-based hash, so any
element of any workload can be regenerated on its own from (seed, role, step, rank,
flat index).  It holds none of the optimizer's arithmetic; tests, the smoke check and
the benchmark use it to feed both the CUDA path and the CPU oracle.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_SRC = os.path.join(HERE, "zsynth_host.c")
DEV_SRC = os.path.join(HERE, "zsynth_dev.cu")
HDR = os.path.join(HERE, "zsynth.h")
HOST_LIB = os.path.join(HERE, "libzsynth_host.so")
DEV_LIB = os.path.join(HERE, "libzsynth_dev.so")

ROLE_GRAD, ROLE_MASTER, ROLE_MOM, ROLE_VAR = 1, 2, 3, 4
NORMAL, NORMAL_SQ, STUDENT_T3 = 0, 1, 2
OUT_F32, OUT_BF16, OUT_F16 = 0, 1, 2

_NP_OUT = {OUT_F32: np.float32, OUT_BF16: np.uint16, OUT_F16: np.uint16}


def _stale(out, *srcs):
    return not os.path.exists(out) or any(os.path.getmtime(out) < os.path.getmtime(s) for s in srcs)


def host_build_cmd(out=HOST_LIB):
    return ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
            "-std=c11", "-o", out, HOST_SRC, "-lm"]


def dev_build_cmd(out=DEV_LIB, arch="sm_103a"):
    cc = arch.replace("sm_", "")
    return ["nvcc", "-O3", "--fmad=false", "-prec-div=true", "-prec-sqrt=true",
            f"-gencode=arch=compute_{cc},code=sm_{cc}", "-Xcompiler", "-fPIC", "-shared",
            "-o", out, DEV_SRC]


def build_host(force=False):
    if force or _stale(HOST_LIB, HOST_SRC, HDR):
        subprocess.run(host_build_cmd(), check=True)
    return HOST_LIB


def build_dev(force=False):
    if force or _stale(DEV_LIB, DEV_SRC, HDR):
        subprocess.run(dev_build_cmd(), check=True)
    return DEV_LIB


_host = None
_dev = None


def host():
    global _host
    if _host is None:
        L = C.CDLL(build_host())
        L.zsynth_key.argtypes = [C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint32]
        L.zsynth_key.restype = C.c_uint64
        L.zsynth_normal.argtypes = [C.c_uint64, C.c_uint64]
        L.zsynth_normal.restype = C.c_float
        L.zsynth_value.argtypes = [C.c_int, C.c_uint64, C.c_uint64, C.c_float, C.c_float]
        L.zsynth_value.restype = C.c_float
        L.zsynth_f32_to_f16.argtypes = [C.c_float]
        L.zsynth_f32_to_f16.restype = C.c_uint16
        L.zsynth_f32_to_bf16.argtypes = [C.c_float]
        L.zsynth_f32_to_bf16.restype = C.c_uint16
        L.zsynth_fill_host.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_uint64, C.c_uint64,
                                       C.c_uint64, C.c_uint64, C.c_float, C.c_float]
        L.zsynth_fill_host.restype = None
        L.zsynth_gather_host.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_uint64, C.c_void_p,
                                         C.c_uint64, C.c_uint64, C.c_float, C.c_float]
        L.zsynth_gather_host.restype = None
        _host = L
    return _host


def dev():
    global _dev
    if _dev is None:
        L = C.CDLL(build_dev())
        L.zsynth_fill_dev.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_uint64, C.c_uint64,
                                      C.c_uint64, C.c_uint64, C.c_float, C.c_float, C.c_void_p,
                                      C.c_int]
        L.zsynth_fill_dev.restype = C.c_int
        _dev = L
    return _dev


def key(seed: int, role: int, step: int = 0, rank: int = 0) -> int:
    return host().zsynth_key(seed, role, step, rank)


def fill_host(out: int, kind: int, k: int, begin: int, count: int, valid_end: int,
              sigma: float, scale: float = 1.0, dst: np.ndarray | None = None) -> np.ndarray:
    if dst is None:
        dst = np.empty(count, dtype=_NP_OUT[out])
    assert dst.dtype == _NP_OUT[out] and dst.size >= count and dst.flags["C_CONTIGUOUS"]
    host().zsynth_fill_host(dst.ctypes.data, out, kind, k, begin, count, valid_end, sigma, scale)
    return dst


def gather_host(out: int, kind: int, k: int, idx: np.ndarray, valid_end: int, sigma: float,
                scale: float = 1.0) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.uint64)
    dst = np.empty(idx.size, dtype=_NP_OUT[out])
    host().zsynth_gather_host(dst.ctypes.data, out, kind, k, idx.ctypes.data, idx.size, valid_end,
                              sigma, scale)
    return dst


def fill_dev(ptr: int, out: int, kind: int, k: int, begin: int, count: int, valid_end: int,
             sigma: float, scale: float = 1.0, stream: int = 0, blocks_per_sm: int = 0) -> None:
    rc = dev().zsynth_fill_dev(ptr, out, kind, k, begin, count, valid_end, sigma, scale, stream,
                               blocks_per_sm)
    if rc != 0:
        raise RuntimeError(f"zsynth_fill_dev failed ({rc})")
