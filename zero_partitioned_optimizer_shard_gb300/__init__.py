"""GB300 ZeRO-DP partitioned mixed-precision AdamW step: Python binding of libzero_shard.so.

Argument marshalling only: every function here converts tensors to raw pointers and the
current CUDA stream to a handle, calls the C entry point of the same name declared in
include/zero.h, and raises ZeroError on a non-zero status.  All computation happens in
the library's CUDA kernels; if the library has not been built, loading fails loudly
(there is no fallback).  Build it with ``zero_partitioned_optimizer_shard_gb300._build.build()``
or ``__graft_entry__.build()``.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libzero_shard.so")

ZERO_OK, ZERO_EINVAL, ZERO_EALIGN, ZERO_ENOMEM, ZERO_ECUDA, ZERO_ETIMEOUT = 0, -1, -2, -3, -4, -5
ZERO_F16, ZERO_BF16 = 1, 2
ZERO_MAX_KERNEL_RANKS = 64
ZERO_TILE_ELEMS = 8192


class ZeroError(RuntimeError):
    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        msg = _lib().zero_strerror(status).decode()
        super().__init__(f"{fn}: {msg} (status {status}" +
                         (f", cudaError {cuda_error})" if status == ZERO_ECUDA else ")"))


class Layout(C.Structure):
    _fields_ = [
        ("psi", C.c_uint64), ("shard", C.c_uint64), ("psi_padded", C.c_uint64), ("pad", C.c_uint64),
        ("bucket_elems", C.c_uint64), ("n_buckets", C.c_uint64), ("tiles_per_rank", C.c_uint64),
        ("n_tiles", C.c_uint64), ("bytes_per_rank", C.c_uint64 * 4),
        ("comm_elems_per_rank", C.c_uint64 * 4), ("n_ranks", C.c_uint32), ("stage", C.c_uint32),
        ("align", C.c_uint32), ("tile_elems", C.c_uint32),
    ]


class HParams(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float), ("eps", C.c_float),
                ("weight_decay", C.c_float), ("max_grad_norm", C.c_float),
                ("params_dtype", C.c_uint32)]


class StepState(C.Structure):
    _fields_ = [
        ("sumsq", C.c_double), ("norm", C.c_double), ("clip_coef", C.c_float),
        ("loss_scale", C.c_float), ("inv_scale", C.c_float), ("step_size", C.c_float),
        ("rbc2", C.c_float), ("decay", C.c_float), ("overflow", C.c_uint32), ("skip", C.c_uint32),
        ("t", C.c_uint32), ("good_steps", C.c_uint32), ("growth_interval", C.c_uint32),
        ("dynamic", C.c_uint32), ("n_ranks", C.c_uint32), ("n_steps", C.c_uint32),
        ("n_skipped", C.c_uint32), ("error", C.c_uint32), ("arrivals", C.c_uint32),
        ("inv_scale_used", C.c_float), ("launch_arrivals", C.c_uint32),
        ("applied_c", C.c_float), ("adamw_next_chunk", C.c_uint64), ("adamw_done", C.c_uint32),
        ("reserved", C.c_uint32 * 5),
    ]


assert C.sizeof(StepState) == 128
STATE_BYTES = C.sizeof(StepState)

_P = C.c_void_p
_L = None


def _lib() -> C.CDLL:
    global _L
    if _L is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                               "(zero_partitioned_optimizer_shard_gb300._build.build())")
        L = C.CDLL(LIB_PATH)
        L.zero_partition.argtypes = [C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint32, C.c_uint64,
                                     C.POINTER(Layout)]
        L.zero_segment_map.argtypes = [C.POINTER(Layout), _P, C.c_uint64, _P, C.c_uint64,
                                       C.POINTER(C.c_uint64)]
        L.zero_workspace_bytes.argtypes = [C.POINTER(Layout)]
        L.zero_workspace_bytes.restype = C.c_size_t
        L.zero_step_state_init.argtypes = [C.POINTER(Layout), C.c_float, C.c_uint32, C.c_uint32,
                                           _P, _P, _P]
        L.zero_step_state_read.argtypes = [_P, C.POINTER(StepState), _P]
        L.zero_step_state_write.argtypes = [_P, C.POINTER(StepState), _P]
        L.zero_reduce_shard_unscale.argtypes = [C.POINTER(Layout), C.c_int, C.POINTER(_P),
                                                C.c_uint64, C.c_uint64, _P, _P, _P, _P]
        L.zero_grad_norm.argtypes = [C.POINTER(Layout), C.POINTER(HParams), _P, _P, _P]
        L.zero_adamw_cast_gather.argtypes = [C.POINTER(Layout), C.POINTER(HParams), _P, _P, _P, _P,
                                             _P, _P, _P]
        L.zero_adamw_cast_gather_host_state.argtypes = L.zero_adamw_cast_gather.argtypes
        L.zero_step.argtypes = [C.POINTER(Layout), C.POINTER(HParams), C.c_int, C.POINTER(_P), _P,
                                _P, _P, _P, _P, _P, _P, _P]
        L.zero_step_host.argtypes = [C.POINTER(Layout), C.POINTER(HParams), C.c_int, C.POINTER(_P),
                                     _P, C.c_uint64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]
        L.zero_reduce_shard_unscale_local.argtypes = [C.POINTER(Layout), C.c_int, C.c_uint32,
                                                      C.c_uint32, C.POINTER(_P), C.c_uint64,
                                                      C.c_uint64, _P, _P, _P, _P]
        L.zero_adamw_cast_gather_local.argtypes = [C.POINTER(Layout), C.POINTER(HParams),
                                                   C.c_uint32, C.c_uint32, _P, _P, _P, _P, _P,
                                                   _P, _P]
        L.zero_step_launches.argtypes = [C.POINTER(Layout), C.c_int]
        L.zero_step_static_workspace.argtypes = [C.POINTER(Layout), C.POINTER(HParams), C.c_int,
                                                 C.POINTER(_P), _P, _P, _P, _P, _P, _P, _P]
        L.zero_strerror.argtypes = [C.c_int]
        L.zero_strerror.restype = C.c_char_p
        L.zero_last_cuda_error.argtypes = []
        for name in ("zero_partition", "zero_segment_map", "zero_step_state_init", "zero_step_state_read",
                     "zero_step_state_write", "zero_reduce_shard_unscale", "zero_grad_norm",
                     "zero_adamw_cast_gather", "zero_adamw_cast_gather_host_state", "zero_step",
                     "zero_step_host", "zero_last_cuda_error", "zero_reduce_shard_unscale_local",
                     "zero_adamw_cast_gather_local", "zero_step_launches",
                     "zero_step_static_workspace"):
            getattr(L, name).restype = C.c_int
        _L = L
    return _L


def lib() -> C.CDLL:
    """The loaded library (raises if it has not been built)."""
    return _lib()


def _check(fn: str, status: int) -> None:
    if status != ZERO_OK:
        raise ZeroError(fn, status, _lib().zero_last_cuda_error() if status == ZERO_ECUDA else 0)


def _ptr(x) -> int | None:
    """Tensor, int address or None -> address."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr_array(xs: Sequence) -> C.Array:
    return (_P * len(xs))(*[_ptr(x) for x in xs])


def hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01,
            max_grad_norm=1.0, params_dtype=0) -> HParams:
    """params_dtype: 0 or ZERO_BF16 for bf16 gathered parameters, ZERO_F16 for fp16."""
    return HParams(lr, beta1, beta2, eps, weight_decay, max_grad_norm, params_dtype)


# --------------------------------------------------------------------------------------
# entry points (same names as include/zero.h)
# --------------------------------------------------------------------------------------
def zero_partition(psi: int, n_ranks: int, stage: int = 2, align: int = 1,
                   bucket_elems: int = 0) -> Layout:
    lay = Layout()
    _check("zero_partition", _lib().zero_partition(psi, n_ranks, stage, align, bucket_elems,
                                                   C.byref(lay)))
    return lay


class Segment(C.Structure):
    """One piece of a model tensor inside one rank's shard (zero_segment_t)."""
    _fields_ = [("tensor", C.c_uint64), ("rank", C.c_uint64), ("tensor_offset", C.c_uint64),
                ("shard_offset", C.c_uint64), ("count", C.c_uint64)]


def zero_segment_map(layout: Layout, tensor_elems: Sequence[int]) -> list:
    """Each tensor's piece on each rank, in flat order: a list of Segment."""
    n_t = len(tensor_elems)
    sizes = (C.c_uint64 * max(n_t, 1))(*tensor_elems)
    n = C.c_uint64()
    _check("zero_segment_map", _lib().zero_segment_map(C.byref(layout), sizes, n_t, None, 0,
                                                       C.byref(n)))
    out = (Segment * max(n.value, 1))()
    _check("zero_segment_map", _lib().zero_segment_map(C.byref(layout), sizes, n_t, out, n.value,
                                                       C.byref(n)))
    return list(out[:n.value])


def zero_workspace_bytes(layout: Layout) -> int:
    return _lib().zero_workspace_bytes(C.byref(layout))


def zero_step_state_init(layout: Layout, loss_scale: float, dynamic: bool, growth_interval: int,
                         st, partials, stream=None) -> None:
    _check("zero_step_state_init", _lib().zero_step_state_init(
        C.byref(layout), loss_scale, int(bool(dynamic)), growth_interval, _ptr(st), _ptr(partials),
        _stream(stream)))


def zero_step_state_read(st, stream=None) -> StepState:
    out = StepState()
    _check("zero_step_state_read", _lib().zero_step_state_read(_ptr(st), C.byref(out), _stream(stream)))
    return out


def zero_step_state_write(st, state: StepState, stream=None) -> None:
    _check("zero_step_state_write", _lib().zero_step_state_write(_ptr(st), C.byref(state),
                                                                 _stream(stream)))


def zero_reduce_shard_unscale(layout: Layout, dtype: int, replicas: Sequence, begin: int, count: int,
                              g, partials, st, stream=None) -> None:
    _check("zero_reduce_shard_unscale", _lib().zero_reduce_shard_unscale(
        C.byref(layout), dtype, _ptr_array(replicas), begin, count, _ptr(g), _ptr(partials),
        _ptr(st), _stream(stream)))


def zero_grad_norm(layout: Layout, hp: HParams, partials, st, stream=None) -> None:
    _check("zero_grad_norm", _lib().zero_grad_norm(C.byref(layout), C.byref(hp), _ptr(partials),
                                                   _ptr(st), _stream(stream)))


def zero_adamw_cast_gather(layout: Layout, hp: HParams, g, master, m, v, params, st,
                           stream=None) -> None:
    _check("zero_adamw_cast_gather", _lib().zero_adamw_cast_gather(
        C.byref(layout), C.byref(hp), _ptr(g), _ptr(master), _ptr(m), _ptr(v), _ptr(params),
        _ptr(st), _stream(stream)))


def zero_adamw_cast_gather_host_state(layout: Layout, hp: HParams, g, master, m, v, params, st,
                                      stream=None) -> None:
    """master, m, v: page-locked host buffers (e.g. torch pin_memory tensors)."""
    _check("zero_adamw_cast_gather_host_state", _lib().zero_adamw_cast_gather_host_state(
        C.byref(layout), C.byref(hp), _ptr(g), _ptr(master), _ptr(m), _ptr(v), _ptr(params),
        _ptr(st), _stream(stream)))


def zero_reduce_shard_unscale_local(layout: Layout, dtype: int, rank_begin: int, rank_count: int,
                                    replicas: Sequence, begin: int, count: int, g_local, partials,
                                    st, stream=None) -> None:
    """g_local holds flat [rank_begin*S, (rank_begin+rank_count)*S) from index 0."""
    f = _lib().zero_reduce_shard_unscale_local
    _check("zero_reduce_shard_unscale_local", f(
        C.byref(layout), dtype, rank_begin, rank_count, _ptr_array(replicas), begin, count,
        _ptr(g_local), _ptr(partials), _ptr(st), _stream(stream)))


def zero_adamw_cast_gather_local(layout: Layout, hp: HParams, rank_begin: int, rank_count: int,
                                 g_local, master_local, m_local, v_local, params_local, st,
                                 stream=None) -> None:
    f = _lib().zero_adamw_cast_gather_local
    _check("zero_adamw_cast_gather_local", f(
        C.byref(layout), C.byref(hp), rank_begin, rank_count, _ptr(g_local), _ptr(master_local),
        _ptr(m_local), _ptr(v_local), _ptr(params_local), _ptr(st), _stream(stream)))


def zero_step(layout: Layout, hp: HParams, dtype: int, replicas: Sequence, g, partials, master, m,
              v, params, st, stream=None) -> None:
    """replicas: n_buckets * N device buffers (or addresses), bucket-major."""
    _check("zero_step", _lib().zero_step(
        C.byref(layout), C.byref(hp), dtype, _ptr_array(replicas), _ptr(g), _ptr(partials),
        _ptr(master), _ptr(m), _ptr(v), _ptr(params), _ptr(st), _stream(stream)))


def zero_step_launches(layout: Layout, dtype: int) -> int:
    """Kernel launches of one zero_step call for this layout: 1 (single-launch step) or
    n_buckets + 2."""
    f = _lib().zero_step_launches
    n = f(C.byref(layout), dtype)
    if n < 0:
        _check("zero_step_launches", n)
    return n


def zero_step_host(layout: Layout, hp: HParams, dtype: int, host_replicas: Sequence, staging,
                   staging_bytes: int, g, partials, master, m, v, params, st,
                   host_state_out=None, stream=None, copy_stream=None) -> None:
    """host_replicas: N pinned host buffers (or addresses) of psi_padded elements each."""
    _check("zero_step_host", _lib().zero_step_host(
        C.byref(layout), C.byref(hp), dtype, _ptr_array(host_replicas), _ptr(staging),
        staging_bytes, _ptr(g), _ptr(partials), _ptr(master), _ptr(m), _ptr(v), _ptr(params),
        _ptr(st), _ptr(host_state_out), _stream(stream), _stream(copy_stream)))


def zero_step_static_workspace(layout: Layout, hp: HParams, dtype: int, replicas: Sequence, g,
                               master, m, v, params, st, stream=None) -> None:
    """zero_step without a caller workspace: for callers that cannot allocate device
    memory.  The per-tile partials live in the library's static device array (8 MiB per
    GPU); calls must not overlap on the GPU.  See include/zero.h."""
    f = _lib().zero_step_static_workspace
    _check("zero_step_static_workspace", f(
        C.byref(layout), C.byref(hp), dtype, _ptr_array(replicas), _ptr(g), _ptr(master), _ptr(m),
        _ptr(v), _ptr(params), _ptr(st), _stream(stream)))


__all__ = [
    "Layout", "HParams", "StepState", "ZeroError", "hparams", "lib", "STATE_BYTES",
    "ZERO_F16", "ZERO_BF16", "Segment", "zero_partition", "zero_segment_map", "zero_workspace_bytes", "zero_step_state_init",
    "zero_step_state_read", "zero_step_state_write", "zero_reduce_shard_unscale",
    "zero_grad_norm", "zero_adamw_cast_gather", "zero_adamw_cast_gather_host_state", "zero_step",
    "zero_step_host", "zero_step_launches", "zero_reduce_shard_unscale_local",
    "zero_adamw_cast_gather_local", "zero_step_static_workspace",
]
