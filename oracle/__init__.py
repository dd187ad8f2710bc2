"""CPU oracle of the ZeRO-DP partitioned mixed-precision AdamW step (ctypes binding).

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH: only the test suite, the smoke check
and the benchmark's CPU-baseline leg import this package.  The C source
(``zero_oracle.c``) is a plain serial restatement of the step, written from the ZeRO
pages; it shares no code with the CUDA library.  numpy arrays in, numpy arrays out.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "zero_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

F16 = 1
BF16 = 2

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-std=c11"]


def build(src: str = SRC, out: str = LIB, force: bool = False) -> str:
    """Compile the oracle with gcc (no fused multiply-add, no fast-math)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


class Layout(C.Structure):
    _fields_ = [
        ("psi", C.c_uint64), ("n_ranks", C.c_uint64), ("shard", C.c_uint64),
        ("psi_padded", C.c_uint64), ("pad", C.c_uint64), ("align", C.c_uint64),
        ("bucket_elems", C.c_uint64), ("n_buckets", C.c_uint64), ("stage", C.c_uint64),
        ("bytes_per_rank", C.c_uint64 * 4), ("comm_elems_per_rank", C.c_uint64 * 4),
    ]


class HParams(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float),
                ("eps", C.c_float), ("weight_decay", C.c_float), ("max_grad_norm", C.c_float),
                ("params_dtype", C.c_uint32)]


class Scaler(C.Structure):
    _fields_ = [("loss_scale", C.c_float), ("dynamic", C.c_uint32),
                ("growth_interval", C.c_uint32), ("good_steps", C.c_uint32),
                ("t", C.c_uint32), ("n_skipped", C.c_uint32)]


class Report(C.Structure):
    _fields_ = [("sumsq", C.c_double), ("norm", C.c_double), ("clip_coef", C.c_float),
                ("loss_scale_used", C.c_float), ("loss_scale_next", C.c_float),
                ("overflow", C.c_uint32), ("skipped", C.c_uint32), ("t", C.c_uint32)]


_P = C.c_void_p


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


@dataclass
class Oracle:
    lib: C.CDLL

    def __post_init__(self):
        L = self.lib
        L.oracle_f16_to_f32.argtypes = [C.c_uint16]
        L.oracle_f16_to_f32.restype = C.c_float
        L.oracle_bf16_to_f32.argtypes = [C.c_uint16]
        L.oracle_bf16_to_f32.restype = C.c_float
        L.oracle_f32_to_bf16.argtypes = [C.c_float]
        L.oracle_f32_to_bf16.restype = C.c_uint16
        L.oracle_f32_to_f16.argtypes = [C.c_float]
        L.oracle_f32_to_f16.restype = C.c_uint16
        L.oracle_partition.argtypes = [C.c_uint64, C.c_uint64, C.c_uint32, C.c_uint64,
                                       C.c_uint64, C.POINTER(Layout)]
        L.oracle_partition.restype = C.c_int
        L.oracle_inv_scale.argtypes = [C.c_uint64, C.c_float]
        L.oracle_inv_scale.restype = C.c_float
        L.oracle_reduce_window.argtypes = [C.POINTER(Layout), C.c_int, _P, C.c_uint64,
                                           C.c_uint64, C.c_float, _P, _P, _P]
        L.oracle_reduce_window.restype = None
        L.oracle_global_norm.argtypes = [_P, C.c_uint64, C.POINTER(C.c_double)]
        L.oracle_global_norm.restype = C.c_double
        L.oracle_clip_coef.argtypes = [C.c_double, C.c_float]
        L.oracle_clip_coef.restype = C.c_float
        L.oracle_scaler_update.argtypes = [C.POINTER(Scaler), C.c_uint32]
        L.oracle_scaler_update.restype = C.c_int
        L.oracle_adamw_scalars.argtypes = [C.POINTER(HParams), C.c_uint32, C.POINTER(C.c_float),
                                           C.POINTER(C.c_float), C.POINTER(C.c_float)]
        L.oracle_adamw_scalars.restype = None
        L.oracle_adamw_elements.argtypes = [C.POINTER(HParams), C.c_float, C.c_uint32,
                                            C.c_uint64, _P, _P, _P, _P, _P]
        L.oracle_adamw_elements.restype = None
        L.oracle_adamw_shard.argtypes = [C.POINTER(Layout), C.POINTER(HParams), C.c_float,
                                         C.c_uint32, C.c_uint64, _P, _P, _P, _P, _P]
        L.oracle_adamw_shard.restype = None
        L.oracle_step.argtypes = [C.POINTER(Layout), C.POINTER(HParams), C.c_int, _P, _P, _P,
                                  _P, _P, _P, C.POINTER(Scaler), C.POINTER(Report)]
        L.oracle_step.restype = C.c_int
        L.oracle_step_unsharded.argtypes = [C.c_uint64, C.POINTER(HParams), _P, _P, _P, _P, _P,
                                            C.POINTER(Scaler), C.POINTER(Report)]
        L.oracle_step_unsharded.restype = C.c_int
        L.oracle_segment_map.argtypes = [C.POINTER(Layout), _P, C.c_uint64, _P, C.c_uint64]
        L.oracle_segment_map.restype = C.c_int64

    # -- number formats ------------------------------------------------------------------
    def f16_to_f32(self, bits: int) -> float:
        return self.lib.oracle_f16_to_f32(bits)

    def bf16_to_f32(self, bits: int) -> float:
        return self.lib.oracle_bf16_to_f32(bits)

    def f32_to_bf16(self, x: float) -> int:
        return self.lib.oracle_f32_to_bf16(x)

    def f32_to_f16(self, x: float) -> int:
        return self.lib.oracle_f32_to_f16(x)

    # -- layout ----------------------------------------------------------------------------
    def partition(self, psi, n_ranks, stage=2, align=1, bucket_elems=0) -> Layout:
        lay = Layout()
        rc = self.lib.oracle_partition(psi, n_ranks, stage, align, bucket_elems, C.byref(lay))
        if rc != 0:
            raise ValueError(f"oracle_partition rejected psi={psi} n={n_ranks} stage={stage}")
        return lay

    def inv_scale(self, n_ranks, loss_scale) -> float:
        return self.lib.oracle_inv_scale(n_ranks, loss_scale)

    # -- reduce ------------------------------------------------------------------------------
    def reduce_window(self, lay, dtype, replicas, begin, count, inv_scale, g, sumsq, overflow):
        """replicas: N uint16 arrays and g: one float32 array, all starting at flat `begin`."""
        assert len(replicas) == lay.n_ranks and g.dtype == np.float32 and g.size >= count
        assert sumsq.dtype == np.float64 and overflow.dtype == np.uint32
        for r in replicas:
            assert r.dtype == np.uint16 and r.size >= count
        ptrs = (C.c_void_p * len(replicas))(*[_ptr(r) for r in replicas])
        self.lib.oracle_reduce_window(C.byref(lay), dtype, ptrs, begin, count, inv_scale,
                                      _ptr(g), _ptr(sumsq), _ptr(overflow))

    def global_norm(self, sumsq: np.ndarray):
        tot = C.c_double()
        n = self.lib.oracle_global_norm(_ptr(sumsq), sumsq.size, C.byref(tot))
        return n, tot.value

    def clip_coef(self, norm: float, max_norm: float) -> float:
        return self.lib.oracle_clip_coef(norm, max_norm)

    # -- scaler / AdamW ---------------------------------------------------------------------
    def scaler_update(self, sc: Scaler, overflow: int) -> int:
        return self.lib.oracle_scaler_update(C.byref(sc), overflow)

    def adamw_scalars(self, hp: HParams, t: int):
        a, b, c = C.c_float(), C.c_float(), C.c_float()
        self.lib.oracle_adamw_scalars(C.byref(hp), t, C.byref(a), C.byref(b), C.byref(c))
        return a.value, b.value, c.value

    def adamw_elements(self, hp, clip_coef, t, g, master, m, v, out):
        n = g.size
        for a in (master, m, v):
            assert a.dtype == np.float32 and a.size == n
        assert out.dtype == np.uint16 and out.size == n
        self.lib.oracle_adamw_elements(C.byref(hp), clip_coef, t, n, _ptr(g), _ptr(master),
                                       _ptr(m), _ptr(v), _ptr(out))

    def adamw_shard(self, lay, hp, clip_coef, t, rank, g, master, m, v, out):
        self.lib.oracle_adamw_shard(C.byref(lay), C.byref(hp), clip_coef, t, rank, _ptr(g),
                                    _ptr(master), _ptr(m), _ptr(v), _ptr(out))

    def step(self, lay, hp, dtype, replicas, g, master, m, v, out, sc) -> Report:
        P = lay.psi_padded
        assert len(replicas) == lay.n_ranks
        for r in replicas:
            assert r.dtype == np.uint16 and r.size == P
        for a in (g, master, m, v):
            assert a.dtype == np.float32 and a.size == P
        assert out.dtype == np.uint16 and out.size == P
        ptrs = (C.c_void_p * len(replicas))(*[_ptr(r) for r in replicas])
        rep = Report()
        rc = self.lib.oracle_step(C.byref(lay), C.byref(hp), dtype, ptrs, _ptr(g), _ptr(master),
                                  _ptr(m), _ptr(v), _ptr(out), C.byref(sc), C.byref(rep))
        if rc != 0:
            raise ValueError("oracle_step rejected its arguments")
        return rep

    def step_unsharded(self, hp, g_mean, master, m, v, out, sc) -> Report:
        rep = Report()
        self.lib.oracle_step_unsharded(g_mean.size, C.byref(hp), _ptr(g_mean), _ptr(master),
                                       _ptr(m), _ptr(v), _ptr(out), C.byref(sc), C.byref(rep))
        return rep

    # -- per-tensor segment map -------------------------------------------------------------
    def segment_map(self, lay, tensor_elems) -> np.ndarray:
        """Rows (tensor, rank, tensor_offset, shard_offset, count), in flat order."""
        sizes = np.ascontiguousarray(tensor_elems, dtype=np.uint64)
        n = self.lib.oracle_segment_map(C.byref(lay), _ptr(sizes) if sizes.size else None,
                                        sizes.size, None, 0)
        if n < 0:
            raise ValueError("tensor sizes do not sum to psi")
        out = np.zeros((max(n, 1), 5), dtype=np.uint64)
        self.lib.oracle_segment_map(C.byref(lay), _ptr(sizes) if sizes.size else None, sizes.size,
                                    _ptr(out), n)
        return out[:n]


_cache: dict[str, Oracle] = {}


def load(path: str | None = None) -> Oracle:
    """Build (if stale) and load the oracle library; `path` loads another build of it."""
    path = path or build()
    if path not in _cache:
        _cache[path] = Oracle(C.CDLL(path))
    return _cache[path]


def hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, max_grad_norm=1.0,
            params_dtype=0):
    return HParams(lr, beta1, beta2, eps, weight_decay, max_grad_norm, params_dtype)


def scaler(loss_scale=1.0, dynamic=False, growth_interval=1000, t=0):
    return Scaler(loss_scale, int(dynamic), growth_interval, 0, t, 0)
