"""Write the oracle's per-step results for the full-size workloads (tests/golden/*_steps.txt).

Calls only the CPU oracle and the seeded input generator.  The full-size workloads are too
large for the oracle to hold in memory, so each step streams the flat buffer in chunks:
the generator regenerates every rank's gradient copy for a chunk, the oracle reduces it
(fp32 rank-ordered sum, unscale, overflow flag, fp64 sum of squares in ascending index
order within the chunk), and the chunk sums of squares are added rank by rank in
ascending chunk order.  Then the oracle's norm, scaler and clip coefficient give the
step's scalars.  Those scalars are all a full-size parity test needs from the oracle:
the AdamW update of any sampled element follows from them and its own inputs.

Usage: python tests/golden/make_golden.py C2 [C3 C5 ...]   (uses every host core)
       python tests/golden/make_golden.py sweep      (every bandwidth-sweep point up to
                                                      2^24+1 parameters, into golden/sweep/)
       python tests/golden/make_golden.py sweep-sampled   (2^27, 2^29, 2^31 and +1 at
                                                      N = 2, 8, 64)
"""
from __future__ import annotations

import multiprocessing as mp
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

CHUNK = 1 << 23


def _worker_init():
    os.environ["OMP_NUM_THREADS"] = "1"
    sys.path.insert(0, ROOT)


def _chunk_job(args):
    wl_name, step, loss_scale, r, j0, j1 = args
    import oracle
    import synth
    from synth import workloads as W
    wl = W.by_name(wl_name)
    orc = oracle.load()
    lay = orc.partition(wl.psi, wl.n_ranks, wl.stage, 1, 0)
    S = lay.shard
    begin, count = r * S + j0, j1 - j0
    reps = []
    inj = wl.injection(step)
    for k in range(wl.n_ranks):
        x = synth.fill_host(wl.grad_out, wl.grad_kind, wl.grad_key(step, k), begin, count, wl.psi,
                            wl.grad_sigma, loss_scale)
        if inj and inj[0] == k and begin <= inj[1] < begin + count:
            x[inj[1] - begin] = inj[2]
        reps.append(x)
    g = np.empty(count, np.float32)
    sumsq = np.zeros(wl.n_ranks, np.float64)
    ov = np.zeros(1, np.uint32)
    dt = oracle.F16 if wl.grad_dtype == "f16" else oracle.BF16
    orc.reduce_window(lay, dt, reps, begin, count, orc.inv_scale(wl.n_ranks, loss_scale), g, sumsq, ov)
    return r, j0, float(sumsq[r]), int(ov[0])


def run(wl_name: str, procs: int) -> str:
    """Compute the workload's rows and write its golden file."""
    from synth import workloads as W
    wl = W.by_name(wl_name)
    lines = golden_rows(wl_name, procs)
    path = golden_path(wl_name)
    os.makedirs(os.path.dirname(path), exist_ok=True)
    with open(path, "w", encoding="utf-8") as f:
        f.write(f"# Oracle per-step results for workload {wl_name}: {wl.name}\n")
        f.write("# Written by tests/golden/make_golden.py (CPU oracle + seeded generator only).\n")
        f.write("# Sums of squares: fp64, ascending index within 2^23-element chunks, chunks in "
                "ascending order per rank, ranks in order.\n")
        f.write("# step loss_scale_used overflow skipped t_after sumsq(hex) norm(hex) "
                "clip_coef(hex) loss_scale_next\n")
        f.write("\n".join(lines) + "\n")
    return path


def golden_rows(wl_name: str, procs: int) -> list:
    """The workload's golden rows, one text line per step (nothing written)."""
    import oracle
    from synth import workloads as W
    wl = W.by_name(wl_name)
    orc = oracle.load()
    lay = orc.partition(wl.psi, wl.n_ranks, wl.stage, 1, 0)
    S = lay.shard
    hp = oracle.hparams(**wl.hp.__dict__)
    sc = oracle.scaler(wl.loss_scale, wl.dynamic, wl.growth_interval, t=0)
    lines = []
    ctx = mp.get_context("spawn")
    with ctx.Pool(procs, initializer=_worker_init) as pool:
        for step in range(1, wl.steps + 1):
            t0 = time.time()
            L = sc.loss_scale
            jobs = [(wl_name, step, L, r, j0, min(j0 + CHUNK, S))
                    for r in range(wl.n_ranks) for j0 in range(0, S, CHUNK)]
            res = pool.map(_chunk_job, jobs, chunksize=1)
            part = {(r, j0): (s, ov) for r, j0, s, ov in res}
            sumsq = np.zeros(wl.n_ranks, np.float64)
            overflow = 0
            for r in range(wl.n_ranks):
                acc = 0.0
                for j0 in range(0, S, CHUNK):
                    s, ov = part[(r, j0)]
                    acc = acc + s
                    overflow |= ov
                sumsq[r] = acc
            norm, total = orc.global_norm(sumsq)
            applied = orc.scaler_update(sc, overflow)
            c = orc.clip_coef(norm, hp.max_grad_norm) if applied else 1.0
            lines.append(f"{step} {L!r} {overflow} {int(not applied)} {sc.t} {total.hex()} "
                         f"{norm.hex()} {float(np.float32(c)).hex()} {sc.loss_scale!r}")
            print(f"[{wl_name}] step {step}: L={L} ov={overflow} norm={norm:.9g} c={c:.9g} "
                  f"t={sc.t} ({time.time() - t0:.0f}s)", flush=True)
    return lines


def golden_path(wl_name: str) -> str:
    sub = ("sweep",) if wl_name.startswith("C4-") else ()
    return os.path.join(ROOT, "tests", "golden", *sub, f"{wl_name}_steps.txt")


def load(wl_name: str):
    """Rows of a golden file as dicts (used by the full-size parity tests)."""
    path = golden_path(wl_name)
    rows = []
    with open(path, encoding="utf-8") as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            s, L, ov, sk, t, q, n, c, Ln = line.split()
            rows.append(dict(step=int(s), loss_scale=float(L), overflow=int(ov), skipped=int(sk),
                             t=int(t), sumsq=float.fromhex(q), norm=float.fromhex(n),
                             clip_coef=float.fromhex(c), loss_scale_next=float(Ln)))
    return rows


if __name__ == "__main__":
    procs = int(os.environ.get("GOLDEN_PROCS", os.cpu_count() or 1))
    for name in sys.argv[1:]:
        if name in ("sweep", "sweep-sampled"):
            from synth import workloads as W
            points = W.SWEEP_PARITY_POINTS if name == "sweep" else W.SWEEP_SAMPLED_POINTS
            for point in points:
                print(run(W.sweep_name(*point), procs))
        else:
            print(run(name, procs))
