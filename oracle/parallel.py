"""The oracle's step on every host core: the timed CPU baseline.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH: only the benchmark's CPU-baseline leg
(and its reference arm) and the tests use it.  The arithmetic is the oracle's own C
functions, unchanged; this module cuts the flat buffer into fixed chunks and runs them on
a pool of spawned worker processes over shared memory:

  phase 1  oracle_reduce_window per chunk (every chunk lies inside one rank's shard): the
           chunk's g, its rank's fp64 sum of squares over the chunk, its overflow flag;
  host     per rank, the chunk sums added in ascending chunk order; then the oracle's
           global_norm, scaler_update and clip_coef (the step's scalars);
  phase 2  oracle_adamw_elements per chunk over the chunk's parameters (padding untouched,
           its gathered value 0).

The chunks are fixed (2^20 elements), so the results do not depend on the number of
worker processes.  The sums of squares are grouped per chunk, so the norm may differ from
the serial oracle_step's in the last bits (both are fp64 sums of the same terms).
"""
from __future__ import annotations

import multiprocessing as mp
import os
import sys
import time
from multiprocessing import shared_memory

import numpy as np

CHUNK = 1 << 20
_W = {}   # per worker: the oracle, the layout, numpy views of the shared arrays


def host_cores() -> int:
    """Cores this process may run on (sched_getaffinity)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _views(names):
    arrs = {}
    shms = {}
    for key, (name, dtype, count) in names.items():
        shm = shared_memory.SharedMemory(name=name)
        shms[key] = shm
        arrs[key] = np.ndarray((count,), dtype=dtype, buffer=shm.buf)
    return arrs, shms


def _init(root, names, P, N, lay_args, hp_args, dtype):
    os.environ["OMP_NUM_THREADS"] = "1"
    if root not in sys.path:
        sys.path.insert(0, root)
    import oracle
    orc = oracle.load()
    _W["orc"] = orc
    _W["lay"] = orc.partition(*lay_args)
    _W["hp"] = oracle.hparams(*hp_args)
    _W["dtype"] = dtype
    _W["arrs"], _W["shms"] = _views(names)


def _fill_job(a):
    """Generate one chunk of every gradient copy and of the state (the seeded recipe)."""
    import synth
    begin, count, grads, states = a
    arrs, psi = _W["arrs"], _W["lay"].psi
    for k, (out, kind, key, sigma, scale) in enumerate(grads):
        arrs["rep"][k * _W["lay"].psi_padded + begin:][:count] = synth.fill_host(
            out, kind, key, begin, count, psi, sigma, scale)
    for name, kind, key, sigma in states:
        if key is None:
            arrs[name][begin:begin + count] = 0
        else:
            arrs[name][begin:begin + count] = synth.fill_host(synth.OUT_F32, kind, key, begin,
                                                             count, psi, sigma)
    return begin


def _reduce_job(a):
    begin, count, inv_scale = a
    lay, arrs = _W["lay"], _W["arrs"]
    P, N = lay.psi_padded, lay.n_ranks
    reps = [arrs["rep"][k * P + begin:k * P + begin + count] for k in range(N)]
    sumsq = np.zeros(N, np.float64)
    ov = np.zeros(1, np.uint32)
    _W["orc"].reduce_window(lay, _W["dtype"], reps, begin, count, inv_scale,
                            arrs["g"][begin:begin + count], sumsq, ov)
    return begin, float(sumsq[begin // lay.shard]), int(ov[0])


def _adamw_job(a):
    begin, count, c, t = a
    arrs = _W["arrs"]
    sl = slice(begin, begin + count)
    _W["orc"].adamw_elements(_W["hp"], c, t, arrs["g"][sl], arrs["master"][sl], arrs["m"][sl],
                             arrs["v"][sl], arrs["out"][sl])
    return begin


class ParallelOracle:
    """The oracle's step of workload `wl` (a synth.workloads.Workload, at its psi) on
    `procs` worker processes.  Gradients are those of step 1, generated once."""

    def __init__(self, wl, procs: int | None = None):
        import oracle
        import synth

        self.wl = wl
        self.procs = procs or host_cores()
        self.orc = oracle.load()
        self.lay = self.orc.partition(wl.psi, wl.n_ranks, wl.stage, 1, 0)
        P, N = self.lay.psi_padded, self.lay.n_ranks
        self.hp = oracle.hparams(**wl.hp.__dict__)
        self.dtype = oracle.F16 if wl.grad_dtype == "f16" else oracle.BF16
        self.sc = oracle.scaler(wl.loss_scale, wl.dynamic, wl.growth_interval)
        spec = {"rep": (np.uint16, N * P), "g": (np.float32, P), "master": (np.float32, P),
                "m": (np.float32, P), "v": (np.float32, P), "out": (np.uint16, P)}
        self._shm = {}
        self.arrs = None
        self.pool = None
        try:
            names = {}
            for key, (dtype, count) in spec.items():
                shm = shared_memory.SharedMemory(create=True,
                                                 size=max(1, count * np.dtype(dtype).itemsize))
                self._shm[key] = shm
                names[key] = (shm.name, dtype, count)
            self.arrs = {k: np.ndarray((c,), dtype=d, buffer=self._shm[k].buf)
                         for k, (d, c) in spec.items()}
            self.arrs["out"][:] = 0
            root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
            lay_args = (wl.psi, wl.n_ranks, wl.stage, 1, 0)
            hp_args = tuple(getattr(self.hp, f) for f, _ in self.hp._fields_)
            self.pool = mp.get_context("spawn").Pool(
                self.procs, initializer=_init,
                initargs=(root, names, P, N, lay_args, hp_args, self.dtype))
            grads = [(wl.grad_out, wl.grad_kind, wl.grad_key(1, k), wl.grad_sigma, wl.loss_scale)
                     for k in range(N)]
            states = [("master", synth.NORMAL, wl.state_key(synth.ROLE_MASTER), wl.master_sigma)]
            if wl.random_moments:
                states += [("m", synth.NORMAL, wl.state_key(synth.ROLE_MOM), wl.mom_sigma),
                           ("v", synth.NORMAL_SQ, wl.state_key(synth.ROLE_VAR), wl.mom_sigma)]
            else:
                states += [("m", None, None, 0.0), ("v", None, None, 0.0)]
            self.pool.map(_fill_job,
                          [(b, min(CHUNK, P - b), grads, states) for b in range(0, P, CHUNK)],
                          chunksize=1)
        except BaseException:
            self.close()  # no shared segment outlives a failed set-up
            raise

    def _chunks(self, lo, hi):
        return [(b, min(CHUNK, hi - b)) for b in range(lo, hi, CHUNK)]

    def step(self) -> dict:
        """One oracle step over the whole buffer; returns its scalars."""
        lay, orc = self.lay, self.orc
        S, N = lay.shard, lay.n_ranks
        inv = orc.inv_scale(N, self.sc.loss_scale)
        jobs = [(b, c, inv) for r in range(N) for b, c in self._chunks(r * S, (r + 1) * S)]
        res = {b: (s, ov) for b, s, ov in self.pool.map(_reduce_job, jobs, chunksize=1)}
        sumsq = np.zeros(N, np.float64)
        overflow = 0
        for r in range(N):
            acc = 0.0
            for b, _ in self._chunks(r * S, (r + 1) * S):
                s, ov = res[b]
                acc = acc + s
                overflow |= ov
            sumsq[r] = acc
        norm, _ = orc.global_norm(sumsq)
        applied = orc.scaler_update(self.sc, overflow)
        c = orc.clip_coef(norm, self.hp.max_grad_norm) if applied else 1.0
        if applied:
            self.pool.map(_adamw_job, [(b, n, c, self.sc.t) for b, n in self._chunks(0, lay.psi)],
                          chunksize=1)
        return {"norm": norm, "clip_coef": c, "overflow": overflow, "t": self.sc.t}

    def time_steps(self, steps: int) -> float:
        """Seconds for `steps` consecutive steps."""
        t0 = time.perf_counter()
        for _ in range(steps):
            self.step()
        return time.perf_counter() - t0

    def close(self) -> None:
        if self.pool is not None:
            self.pool.close()
            self.pool.join()
            self.pool = None
        self.arrs = None
        for shm in self._shm.values():
            shm.close()
            shm.unlink()
        self._shm = {}

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
