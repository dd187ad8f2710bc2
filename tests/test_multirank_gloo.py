"""The ZeRO step across real processes (torch.distributed, gloo, CPU): one process per rank.

Every rank holds its own gradient copy of the whole flat buffer and only its own shard of
the fp32 master/m/v state, as ZeRO-2 prescribes ("【论文解读】ZeRO" sec. 4(2), 6(2)):
  1. reduce-scatter: rank r receives every rank's copy of shard r and averages it (here
     an all-gather of the copies followed by the rank-ordered sum, the same arithmetic
     the single-GPU kernels use);
  2. the global-norm all-reduce (the Megatron page, sec. 1): the per-rank sums of squares
     and overflow flags are all-gathered and added in rank order;
  3. each rank applies AdamW to its own shard, then the bf16 shards are all-gathered into
     the full parameter vector.
The gathered parameters, the norm and every rank's shard state must equal the
single-process oracle's bit for bit.  World size 4 uses the pages' 8-parameter, 4-GPU
example shape as one of its cases.  No GPU is used.
"""
import os
import queue
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import synth

SIGMA = 1e-3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _state(role, kind, sig, begin, count, psi, seed):
    return synth.fill_host(synth.OUT_F32, kind, synth.key(seed, role), begin, count, psi, sig)


def _rank_main(rank, world, port, psi, seed, steps, clip, out_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        orc = oracle.load()
        lay = orc.partition(psi, world, 2)
        S, P = lay.shard, lay.psi_padded
        lo = rank * S
        hp = oracle.hparams(max_grad_norm=clip)
        sc = oracle.scaler(1.0, False)
        # this rank's shard of the optimizer state, laid out at its flat offsets
        master = np.zeros(P, np.float32)
        m = np.zeros(P, np.float32)
        v = np.zeros(P, np.float32)
        master[lo:lo + S] = _state(synth.ROLE_MASTER, synth.NORMAL, 0.02, lo, S, psi, seed)
        m[lo:lo + S] = _state(synth.ROLE_MOM, synth.NORMAL, 1e-4, lo, S, psi, seed)
        v[lo:lo + S] = _state(synth.ROLE_VAR, synth.NORMAL_SQ, 1e-4, lo, S, psi, seed)
        g = np.zeros(P, np.float32)
        out = np.zeros(P, np.uint16)
        results = []
        for step in range(1, steps + 1):
            mine = synth.fill_host(synth.OUT_BF16, synth.NORMAL,
                                   synth.key(seed, synth.ROLE_GRAD, step, rank), 0, P, psi, SIGMA)
            # gloo has no 16-bit collectives: the bit patterns travel as int32
            copies = [torch.empty(P, dtype=torch.int32) for _ in range(world)]
            dist.all_gather(copies, torch.from_numpy(mine.astype(np.int32)))
            shard_copies = [c.numpy()[lo:lo + S].astype(np.uint16) for c in copies]
            sumsq = np.zeros(world, np.float64)
            ov = np.zeros(1, np.uint32)
            orc.reduce_window(lay, oracle.BF16, shard_copies, lo, S, orc.inv_scale(world, 1.0),
                              g[lo:lo + S], sumsq, ov)
            parts = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
            dist.all_gather(parts, torch.tensor([sumsq[rank], float(ov[0])], dtype=torch.float64))
            q = np.array([float(p[0]) for p in parts])
            overflow = int(any(float(p[1]) != 0.0 for p in parts))
            norm, _ = orc.global_norm(q)
            applied = orc.scaler_update(sc, overflow)
            c = orc.clip_coef(norm, hp.max_grad_norm) if applied else 1.0
            if applied:
                orc.adamw_shard(lay, hp, c, sc.t, rank, g, master, m, v, out)
            shards = [torch.empty(S, dtype=torch.int32) for _ in range(world)]
            dist.all_gather(shards, torch.from_numpy(out[lo:lo + S].astype(np.int32)))
            gathered = np.concatenate([t.numpy().astype(np.uint16) for t in shards])
            results.append((norm, c, gathered))
        out_q.put((rank, results, master[lo:lo + S].copy(), m[lo:lo + S].copy(),
                   v[lo:lo + S].copy(), g[lo:lo + S].copy()))
    finally:
        dist.destroy_process_group()


def _single_process(world, psi, seed, steps, clip):
    orc = oracle.load()
    lay = orc.partition(psi, world, 2)
    P = lay.psi_padded
    hp = oracle.hparams(max_grad_norm=clip)
    sc = oracle.scaler(1.0, False)
    master = _state(synth.ROLE_MASTER, synth.NORMAL, 0.02, 0, P, psi, seed)
    m = _state(synth.ROLE_MOM, synth.NORMAL, 1e-4, 0, P, psi, seed)
    v = _state(synth.ROLE_VAR, synth.NORMAL_SQ, 1e-4, 0, P, psi, seed)
    g = np.zeros(P, np.float32)
    out = np.zeros(P, np.uint16)
    res = []
    for step in range(1, steps + 1):
        reps = [synth.fill_host(synth.OUT_BF16, synth.NORMAL,
                                synth.key(seed, synth.ROLE_GRAD, step, k), 0, P, psi, SIGMA)
                for k in range(world)]
        rep = orc.step(lay, hp, oracle.BF16, reps, g, master, m, v, out, sc)
        res.append((rep.norm, rep.clip_coef, out.copy()))
    return lay, res, master, m, v, g


@pytest.mark.parametrize("world,psi,clip", [(2, 10_001, 1e-3), (4, 8, 0.0), (4, 333, 1.0)])
def test_ranks_as_processes_match_single_process(world, psi, clip):
    seed, steps = 11, 3
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, psi, seed, steps, clip, q))
             for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    try:
        for _ in range(world):
            rank, results, master, m, v, g = q.get(timeout=300)
            got[rank] = (results, master, m, v, g)
    except queue.Empty:
        pytest.fail(f"ranks {sorted(set(range(world)) - set(got))} returned nothing")
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.terminate()
    assert all(p.exitcode == 0 for p in procs)
    lay, ref, master, m, v, g = _single_process(world, psi, seed, steps, clip)
    S = lay.shard
    for r in range(world):
        results, ms, mm, mv, mg = got[r]
        for (n_a, c_a, out_a), (n_b, c_b, out_b) in zip(results, ref):
            assert n_a == n_b and c_a == c_b
            assert np.array_equal(out_a, out_b)
        sl = slice(r * S, (r + 1) * S)
        for a, b in ((ms, master[sl]), (mm, m[sl]), (mv, v[sl]), (mg, g[sl])):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


# ---------------------------------------------------------------------------------------
# The product's exchange layer (zero_partitioned_optimizer_shard_gb300.ranks) on CPU: each
# process holds a contiguous group of ranks; the arithmetic of each step is the oracle's,
# the data movement is the library's Exchange (all-to-all of the 16-bit copies, all-gather
# of the per-rank sums of squares and of the parameters, maximum of the overflow word).
# ---------------------------------------------------------------------------------------
def _group_main(proc, world, port, n_ranks, psi, seed, steps, clip, inject, out_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=proc, world_size=world)
    try:
        from zero_partitioned_optimizer_shard_gb300.ranks import Exchange, local_ranks
        ex = Exchange()
        rb, R = local_ranks(n_ranks, world, proc)
        orc = oracle.load()
        lay = orc.partition(psi, n_ranks, 2, 8)
        S, P = lay.shard, lay.psi_padded
        lo, L = rb * S, R * S
        hp = oracle.hparams(max_grad_norm=clip)
        sc = oracle.scaler(1.0, False)
        master = _state(synth.ROLE_MASTER, synth.NORMAL, 0.02, lo, L, psi, seed)
        m = _state(synth.ROLE_MOM, synth.NORMAL, 1e-4, lo, L, psi, seed)
        v = _state(synth.ROLE_VAR, synth.NORMAL_SQ, 1e-4, lo, L, psi, seed)
        g = np.zeros(L, np.float32)
        params = torch.zeros(P, dtype=torch.int16)
        results = []
        for step in range(1, steps + 1):
            copies = []
            for j in range(R):
                c = synth.fill_host(synth.OUT_BF16, synth.NORMAL,
                                    synth.key(seed, synth.ROLE_GRAD, step, rb + j), 0, P, psi, SIGMA)
                if inject and inject[0] == step and inject[1] == rb + j:
                    c[inject[2]] = 0x7F80  # bf16 +inf
                copies.append(torch.from_numpy(c.view(np.int16)))
            recv = [torch.empty(P, dtype=torch.int16) for _ in range(R)]
            for j in range(R):
                ex.all_to_all(recv[j], copies[j])
            # rank k's copy of this process's range: chunk k // R of local copy k % R
            win = [recv[k % R][(k // R) * L:(k // R + 1) * L].numpy().view(np.uint16).copy()
                   for k in range(n_ranks)]
            sumsq = torch.zeros(n_ranks, dtype=torch.float64)
            ov = np.zeros(1, np.uint32)
            orc.reduce_window(lay, oracle.BF16, win, lo, L, orc.inv_scale(n_ranks, 1.0), g,
                              sumsq.numpy(), ov)
            ex.all_gather(sumsq, rb, rb + R)
            flag = torch.tensor([int(ov[0])], dtype=torch.int32)
            ex.maximum(flag)
            norm, _ = orc.global_norm(sumsq.numpy())
            applied = orc.scaler_update(sc, int(flag.item()))
            c = orc.clip_coef(norm, hp.max_grad_norm) if applied else 1.0
            if applied:
                n = max(0, min(L, psi - lo))  # parameters in this range; the rest is padding
                out = np.zeros(L, np.uint16)
                orc.adamw_elements(hp, c, sc.t, g[:n], master[:n], m[:n], v[:n], out[:n])
                params[lo:lo + L] = torch.from_numpy(out.view(np.int16))
                ex.all_gather(params, lo, lo + L)
            results.append((norm, c, int(flag.item()), params.numpy().view(np.uint16).copy()))
        out_q.put((proc, results, master.copy(), m.copy(), v.copy(), g.copy()))
    finally:
        dist.destroy_process_group()


def _single_process_aligned(n_ranks, psi, seed, steps, clip, inject):
    orc = oracle.load()
    lay = orc.partition(psi, n_ranks, 2, 8)
    P = lay.psi_padded
    hp = oracle.hparams(max_grad_norm=clip)
    sc = oracle.scaler(1.0, False)
    master = _state(synth.ROLE_MASTER, synth.NORMAL, 0.02, 0, P, psi, seed)
    m = _state(synth.ROLE_MOM, synth.NORMAL, 1e-4, 0, P, psi, seed)
    v = _state(synth.ROLE_VAR, synth.NORMAL_SQ, 1e-4, 0, P, psi, seed)
    g = np.zeros(P, np.float32)
    out = np.zeros(P, np.uint16)
    res = []
    for step in range(1, steps + 1):
        reps = [synth.fill_host(synth.OUT_BF16, synth.NORMAL,
                                synth.key(seed, synth.ROLE_GRAD, step, k), 0, P, psi, SIGMA)
                for k in range(n_ranks)]
        if inject and inject[0] == step:
            reps[inject[1]][inject[2]] = 0x7F80
        rep = orc.step(lay, hp, oracle.BF16, reps, g, master, m, v, out, sc)
        res.append((rep.norm, rep.clip_coef, rep.overflow, out.copy()))
    return lay, res, master, m, v, g


@pytest.mark.parametrize("world,n_ranks,psi,clip,inject", [
    (2, 2, 10_001, 1e-3, None),
    (2, 4, 5_000, 1.0, (2, 3, 77)),        # two ranks per process; rank 3 overflows at step 2
    (4, 8, 20_011, 1e-3, None),            # two ranks per process, four processes
    (4, 4, 13, 0.0, None),                 # the last ranks hold only padding
])
def test_exchange_layer_over_processes_matches_single_process(world, n_ranks, psi, clip, inject):
    seed, steps = 7, 3
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_group_main,
                         args=(p, world, port, n_ranks, psi, seed, steps, clip, inject, q))
             for p in range(world)]
    for p in procs:
        p.start()
    got = {}
    try:
        for _ in range(world):
            proc, results, master, m, v, g = q.get(timeout=300)
            got[proc] = (results, master, m, v, g)
    except queue.Empty:
        pytest.fail(f"processes {sorted(set(range(world)) - set(got))} returned nothing")
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.terminate()
    assert all(p.exitcode == 0 for p in procs)
    lay, ref, master, m, v, g = _single_process_aligned(n_ranks, psi, seed, steps, clip, inject)
    L = lay.shard * (n_ranks // world)
    for p in range(world):
        results, ms, mm, mv, mg = got[p]
        for (n_a, c_a, f_a, out_a), (n_b, c_b, f_b, out_b) in zip(results, ref):
            assert f_a == f_b
            if not f_b:
                assert n_a == n_b and c_a == c_b
            assert np.array_equal(out_a, out_b)
        sl = slice(p * L, (p + 1) * L)
        for a, b in ((ms, master[sl]), (mm, m[sl]), (mv, v[sl])):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
        # g: bit for bit, NaN payloads aside (an overflowing step's g holds inf/NaN)
        same = (mg.view(np.uint32) == g[sl].view(np.uint32)) | (np.isnan(mg) & np.isnan(g[sl]))
        assert same.all()
    if inject:
        assert any(r[2] for r in ref)  # the injected step really overflowed and was skipped


# ---------------------------------------------------------------------------------------
# A process that leaves between steps: the others learn of it on the host.  The exchange
# layer waits on no flag of its own; its collectives are torch.distributed's, so a peer
# that is gone ends the next collective with an error (connection closed, or the process
# group's timeout), never a hang.  No GPU is involved.
# ---------------------------------------------------------------------------------------
def _leaver_main(proc, world, port, out_q):
    import datetime
    import time

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=proc, world_size=world,
                            timeout=datetime.timedelta(seconds=10))
    from zero_partitioned_optimizer_shard_gb300.ranks import Exchange
    ex = Exchange()
    full = torch.zeros(4 * world, dtype=torch.float64)
    full[4 * proc:4 * proc + 4] = proc + 1
    ex.all_gather(full, 4 * proc, 4 * proc + 4)  # step 1: everyone present
    ok = bool(torch.all(full == torch.arange(world, dtype=torch.float64).repeat_interleave(4) + 1))
    if proc == world - 1:
        out_q.put((proc, ok, "left"))
        out_q.close()
        out_q.join_thread()  # the message is out before the process goes
        os._exit(0)  # leaves between steps, with nothing in flight
    t0 = time.time()
    try:
        flag = torch.tensor([0], dtype=torch.int32)
        ex.maximum(flag)  # step 2: the peer is gone
        out_q.put((proc, ok, "no error"))
    except Exception as e:  # noqa: BLE001 - any collective error is the signal
        out_q.put((proc, ok, f"error after {time.time() - t0:.1f}s: {type(e).__name__}"))
    out_q.close()
    out_q.join_thread()
    os._exit(0)


def test_a_process_that_leaves_ends_the_next_exchange_with_an_error():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_leaver_main, args=(p, world, port, q)) for p in range(world)]
    for p in procs:
        p.start()
    got = {}
    try:
        for _ in range(world):
            proc, ok, what = q.get(timeout=120)
            got[proc] = (ok, what)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.terminate()
    assert got[1] == (True, "left")
    ok, what = got[0]
    assert ok and what.startswith("error after"), what
    assert float(what.split()[2].rstrip("s:")) < 30


# ---------------------------------------------------------------------------------------
# The windowed gradient exchange RankStep makes (ranks.exchange_windows, exchange_plan,
# Exchange.send_recv: point-to-point, two receive slots, the next windows in flight while
# one is reduced), run on CPU tensors with the oracle's arithmetic in place of the kernels.
# ---------------------------------------------------------------------------------------
def _windowed_main(proc, world, port, n_ranks, psi, seed, steps, w, out_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=proc, world_size=world)
    try:
        from zero_partitioned_optimizer_shard_gb300.ranks import (Exchange, exchange_plan,
                                                                   exchange_windows, local_ranks)
        ex = Exchange()
        rb, R = local_ranks(n_ranks, world, proc)
        orc = oracle.load()
        lay = orc.partition(psi, n_ranks, 2, 8)
        S, P = lay.shard, lay.psi_padded
        lo, L = rb * S, R * S
        wins = exchange_windows(L, world, w)
        part = max(c for ws in wins for _, c in ws)
        K = max(len(ws) for ws in wins)
        slots = 2 if K > 1 else 1
        recv = [[torch.zeros(world * part, dtype=torch.int16) for _ in range(R)] for _ in range(slots)]
        hp = oracle.hparams(max_grad_norm=1e-3)
        sc = oracle.scaler(1.0, False)
        master = _state(synth.ROLE_MASTER, synth.NORMAL, 0.02, lo, L, psi, seed)
        m = _state(synth.ROLE_MOM, synth.NORMAL, 1e-4, lo, L, psi, seed)
        v = _state(synth.ROLE_VAR, synth.NORMAL_SQ, 1e-4, lo, L, psi, seed)
        g = np.zeros(L, np.float32)
        params = torch.zeros(P, dtype=torch.int16)
        results = []
        for step in range(1, steps + 1):
            copies = [torch.from_numpy(synth.fill_host(
                synth.OUT_BF16, synth.NORMAL, synth.key(seed, synth.ROLE_GRAD, step, rb + j),
                0, P, psi, SIGMA).view(np.int16)) for j in range(R)]

            def issue(k):
                rv = recv[k % slots]
                sends, recvs = exchange_plan(wins, proc, k, R, part)
                return ex.send_recv([(q, copies[j][b:b + n]) for q, j, b, n in sends],
                                    [(q, rv[j][o:o + n]) for q, j, o, n in recvs])

            sumsq = np.zeros(n_ranks, np.float64)
            ov = np.zeros(1, np.uint32)
            pending = {k: issue(k) for k in range(min(slots, K))}
            for k in range(K):
                if k in pending:
                    pending.pop(k).wait()
                if k < len(wins[proc]):
                    b, n = wins[proc][k]
                    rv = recv[k % slots]
                    reps = []
                    for i in range(n_ranks):  # rank i's copy of this window, in rank order
                        q, j = divmod(i, R)
                        src = copies[j][b:b + n] if q == proc else rv[j][q * part:q * part + n]
                        reps.append(src.numpy().view(np.uint16).copy())
                    orc.reduce_window(lay, oracle.BF16, reps, b, n, orc.inv_scale(n_ranks, 1.0),
                                      g[b - lo:], sumsq, ov)
                if k + slots < K:
                    pending[k + slots] = issue(k + slots)
            ex.all_gather(torch.from_numpy(sumsq), rb, rb + R)  # the norm's inputs
            flag = torch.tensor([int(ov[0])], dtype=torch.int32)
            ex.maximum(flag)
            norm, _ = orc.global_norm(sumsq)
            applied = orc.scaler_update(sc, int(flag.item()))
            c = orc.clip_coef(norm, hp.max_grad_norm) if applied else 1.0
            if applied:
                n = max(0, min(L, psi - lo))
                out = np.zeros(L, np.uint16)
                orc.adamw_elements(hp, c, sc.t, g[:n], master[:n], m[:n], v[:n], out[:n])
                params[lo:lo + L] = torch.from_numpy(out.view(np.int16))
                ex.all_gather(params, lo, lo + L)
            results.append((norm, c, params.numpy().view(np.uint16).copy()))
        out_q.put((proc, results, master.copy(), m.copy(), v.copy(), g.copy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,n_ranks,psi,w", [
    (2, 2, 48_761, 8192),      # 3 and 4 windows on the two processes
    (2, 4, 100_003, 8192),     # two ranks per process
    (4, 8, 200_003, 16384),
    (2, 2, 30_001, 0),         # one window per range
])
def test_windowed_exchange_matches_single_process(world, n_ranks, psi, w):
    seed, steps = 5, 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_windowed_main,
                         args=(p, world, port, n_ranks, psi, seed, steps, w, q))
             for p in range(world)]
    for p in procs:
        p.start()
    got = {}
    try:
        for _ in range(world):
            proc, results, master, m, v, g = q.get(timeout=300)
            got[proc] = (results, master, m, v, g)
    except queue.Empty:
        pytest.fail(f"processes {sorted(set(range(world)) - set(got))} returned nothing")
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.terminate()
    assert all(p.exitcode == 0 for p in procs)
    orc = oracle.load()
    lay = orc.partition(psi, n_ranks, 2, 8)
    P = lay.psi_padded
    hp = oracle.hparams(max_grad_norm=1e-3)
    sc = oracle.scaler(1.0, False)
    master = _state(synth.ROLE_MASTER, synth.NORMAL, 0.02, 0, P, psi, seed)
    m = _state(synth.ROLE_MOM, synth.NORMAL, 1e-4, 0, P, psi, seed)
    v = _state(synth.ROLE_VAR, synth.NORMAL_SQ, 1e-4, 0, P, psi, seed)
    g, out = np.zeros(P, np.float32), np.zeros(P, np.uint16)
    L = lay.shard * (n_ranks // world)
    for step in range(1, steps + 1):
        reps = [synth.fill_host(synth.OUT_BF16, synth.NORMAL,
                                synth.key(seed, synth.ROLE_GRAD, step, k), 0, P, psi, SIGMA)
                for k in range(n_ranks)]
        rep = orc.step(lay, hp, oracle.BF16, reps, g, master, m, v, out, sc)
        for p in range(world):
            n_a, c_a, out_a = got[p][0][step - 1]
            assert n_a == rep.norm and c_a == rep.clip_coef
            assert np.array_equal(out_a, out)
    for p in range(world):
        _, ms, mm, mv, mg = got[p]
        sl = slice(p * L, (p + 1) * L)
        for a, b in ((ms, master[sl]), (mm, m[sl]), (mv, v[sl]), (mg, g[sl])):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
