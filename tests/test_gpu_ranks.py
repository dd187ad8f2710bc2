"""The ZeRO step with its ranks spread over processes, on the GPU.

Each process holds a contiguous group of the N ranks ("【论文解读】ZeRO" sec. 6(2): rank r
keeps and updates only partition r) and runs its part of the step through the C ABI:
zero_reduce_shard_unscale_local over its own flat range, zero_grad_norm after the
all-gather of every process's tile partials and the maximum of the overflow word (the
Megatron page, sec. 1: one all-reduce before clipping), zero_adamw_cast_gather_local, and
the all-gather of the parameters.  The processes share this one GPU; their data plane is
gloo through host memory (zero_partitioned_optimizer_shard_gb300.ranks.Exchange).  No
kernel waits on another process: every exchange happens on the host between launches.

Every process's g, master, m and v, the gathered parameters and the whole 128-byte step
state must equal the one-GPU step on the same layout bit for bit after every step, and
the oracle within the stated tolerances.  The schedule is the one
tests/test_multirank_gloo.py runs with the oracle's arithmetic on CPU.
"""
import os
import queue
import socket
from dataclasses import replace

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import synth
from synth import workloads as W
from tests.gpu_harness import GpuRun, OracleRun, assert_scalars, assert_state_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _proc_main(proc, world, port, wl, bucket, out_q):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=proc, world_size=world)
    try:
        import zero_partitioned_optimizer_shard_gb300 as z
        from zero_partitioned_optimizer_shard_gb300.ranks import RankStep, layout_for

        torch.cuda.set_device(0)
        dev = torch.device("cuda", 0)
        s = torch.cuda.current_stream(dev).cuda_stream
        lay = layout_for(wl.psi, wl.n_ranks, wl.stage, bucket)
        dt = z.ZERO_F16 if wl.grad_dtype == "f16" else z.ZERO_BF16
        rs = RankStep(lay, z.hparams(**wl.hp.__dict__), dt, wl.loss_scale, wl.dynamic,
                      wl.growth_interval, dev, exchange_elems=bucket)
        fills = [(rs.master, synth.ROLE_MASTER, synth.NORMAL, wl.master_sigma)]
        if wl.random_moments:
            fills += [(rs.m, synth.ROLE_MOM, synth.NORMAL, wl.mom_sigma),
                      (rs.v, synth.ROLE_VAR, synth.NORMAL_SQ, wl.mom_sigma)]
        for t_, role, kind, sig in fills:
            synth.fill_dev(t_.data_ptr(), synth.OUT_F32, kind, wl.state_key(role), rs.origin,
                           rs.local_len, wl.psi, sig, 1.0, s)
        P = lay.psi_padded
        copies = [torch.empty(P, dtype=torch.int16, device=dev) for _ in range(rs.rank_count)]
        per_step = []
        for step in range(1, wl.steps + 1):
            L = z.zero_step_state_read(rs.st).loss_scale
            for j, c in enumerate(copies):
                synth.fill_dev(c.data_ptr(), wl.grad_out, wl.grad_kind,
                               wl.grad_key(step, rs.rank_begin + j), 0, P, wl.psi, wl.grad_sigma,
                               L, s)
            inj = wl.injection(step)
            if inj and rs.rank_begin <= inj[0] < rs.rank_begin + rs.rank_count:
                copies[inj[0] - rs.rank_begin][inj[1]] = int(np.uint16(inj[2]).view(np.int16))
            rs.step(copies)
            torch.cuda.synchronize(dev)
            per_step.append((rs.st.cpu().numpy().copy(), rs.params.cpu().numpy().view(np.uint16).copy()))
        out_q.put((proc, rs.origin, rs.local_len, per_step, rs.g.cpu().numpy().copy(),
                   rs.master.cpu().numpy().copy(), rs.m.cpu().numpy().copy(),
                   rs.v.cpu().numpy().copy()))
    finally:
        dist.destroy_process_group()


C5_SMALL = replace(W.scaled(W.C5, 3 * 8192 * 4 + 1001, steps=5), n_ranks=4, inject_every=2,
                   inject_rank=3, inject_base=3 * 8192 * 3 + 17)


@pytest.mark.parametrize("world,wl,bucket", [
    # two ranks, one per process; a ragged last shard
    (2, replace(W.scaled(W.C2, 2 * 5 * 8192 + 1003, steps=3), n_ranks=2), 0),
    # fp16 with a dynamic loss scale, two ranks per process: rank 3's copy overflows on
    # every second step (in process 1's range), so both processes must skip that step
    (2, C5_SMALL, 0),
    # four processes of two ranks each: 2^16-element buckets on the one GPU, 2^16-element
    # exchange windows across the processes (4 windows each)
    (4, replace(W.scaled(W.C2, 8 * 3 * 8192 + 4099, steps=3), n_ranks=8), 1 << 16),
    # a larger buffer: 4.2M parameters, two processes of four ranks, 2^20-element windows
    (2, replace(W.scaled(W.C2, (1 << 22) + 13, steps=2), n_ranks=8), 1 << 20),
    # windows of 8192 elements: the processes hold different numbers of windows (their
    # ranges start at different places of the grid), some exchanges are one-sided
    (2, replace(W.scaled(W.C2, 48_761, steps=2), n_ranks=2), 8192),
    # 13 parameters over 4 ranks of 8 (align 8): process 1 holds only padding
    (2, replace(W.scaled(W.C2, 13, steps=2), n_ranks=4), 0),
    # fp16 gathered parameters
    (2, replace(W.scaled(W.C2, 3 * 8192 * 4 + 77, steps=2), n_ranks=4,
                hp=W.HP(params_dtype=1)), 0),
])
def test_ranks_over_processes_equal_the_one_gpu_step(world, wl, bucket):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_proc_main, args=(p, world, port, wl, bucket, q))
             for p in range(world)]
    for p in procs:
        p.start()
    got = {}
    try:
        for _ in range(world):
            r = q.get(timeout=600)
            got[r[0]] = r[1:]
    except queue.Empty:
        pytest.fail(f"processes {sorted(set(range(world)) - set(got))} returned nothing")
    finally:
        for p in procs:
            p.join(timeout=120)
            if p.is_alive():
                p.terminate()
    assert all(p.exitcode == 0 for p in procs)

    # the one-GPU step on the same layout (three launches per step), and the oracle
    ref = GpuRun(wl, bucket, split=True, align=8)
    orc = OracleRun(wl, align=8)
    skipped = 0
    for step in range(1, wl.steps + 1):
        sr = ref.step(step)
        rep = orc.step(step)
        skipped += rep.skipped
        want_state = ref.st.cpu().numpy()
        want_params = ref.out.cpu().numpy().view(np.uint16)
        for p in range(world):
            st_p, params_p = got[p][2][step - 1]
            assert np.array_equal(st_p, want_state), f"process {p}, step {step}: step state"
            assert np.array_equal(params_p, want_params), f"process {p}, step {step}: parameters"
        assert_scalars(sr, rep)
    if wl.inject_every:
        assert skipped >= 2
    arrays = ref.arrays()
    full = {k: np.empty_like(arrays[k]) for k in ("g", "master", "m", "v")}
    for p in range(world):
        origin, n, _, g, master, m, v = got[p]
        sl = slice(origin, origin + n)
        for k, a in (("g", g), ("master", master), ("m", m), ("v", v)):
            b = arrays[k][sl]
            same = (a.view(np.uint32) == b.view(np.uint32)) | (np.isnan(a) & np.isnan(b))
            assert same.all(), f"process {p}: {k} differs from the one-GPU step"
            full[k][sl] = a
    full["out"] = got[0][2][-1][1]
    assert_state_close(full, orc.arrays(), wl.psi, exact_expected=False)
    ref.check_guards()


def test_exchange_nccl_branch_in_a_one_process_group(monkeypatch):
    """The exchange layer's NCCL branch (collectives on the device tensors themselves, no
    host staging) in a group of one process: NCCL runs every call, so the device views,
    element types and contiguity the branch hands it are exercised, and each call must
    leave its data as a one-process exchange does.  (NCCL takes one process per GPU, so
    the exchange between processes itself runs over gloo in the other tests here.)"""
    import datetime
    import torch.distributed as dist

    import zero_partitioned_optimizer_shard_gb300 as z
    from zero_partitioned_optimizer_shard_gb300.ranks import OVERFLOW_WORD, Exchange, RankStep, layout_for

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(_free_port())
    monkeypatch.setenv("NCCL_SOCKET_IFNAME", "lo")  # one process: the loopback is enough
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if not dist.is_nccl_available():
        pytest.skip("this torch build has no NCCL")
    dist.init_process_group("nccl", rank=0, world_size=1, timeout=datetime.timedelta(seconds=60))
    try:
        ex = Exchange()
        assert ex.nccl and ex.world == 1 and ex.proc == 0
        g = torch.Generator(device="cpu").manual_seed(5)
        params = torch.randint(-32768, 32767, (4 * 1003,), dtype=torch.int16, generator=g).to(dev)
        want = params.clone()
        ex.all_gather(params, 0, params.numel())  # 16-bit data travels as bytes
        assert torch.equal(params, want)
        partials = torch.rand(77, dtype=torch.float64, generator=g).to(dev)
        want = partials.clone()
        ex.all_gather(partials, 0, 77)
        assert torch.equal(partials, want)
        st = torch.zeros(z.STATE_BYTES, dtype=torch.uint8, device=dev)
        st.view(torch.int32)[OVERFLOW_WORD] = 1
        ex.maximum(st.view(torch.int32)[OVERFLOW_WORD:OVERFLOW_WORD + 1])
        assert int(st.view(torch.int32)[OVERFLOW_WORD]) == 1 and int(st.sum()) == 1
        inp = torch.randint(-32768, 32767, (2 * 4096,), dtype=torch.int16, generator=g).to(dev)
        out = torch.empty_like(inp)
        ex.all_to_all(out, inp, [inp.numel()], [inp.numel()], async_op=True).wait()
        assert torch.equal(out, inp)
        ex.send_recv([], []).wait()  # nothing to exchange
        # the step itself through the NCCL group: one process holding all four ranks
        lay = layout_for(100_000, 4)
        rs = RankStep(lay, z.hparams(), z.ZERO_BF16, device=dev)
        copies = [torch.zeros(lay.psi_padded, dtype=torch.int16, device=dev) for _ in range(4)]
        rs.step(copies)
        torch.cuda.synchronize()
        s = z.zero_step_state_read(rs.st)
        assert s.t == 1 and s.norm == 0.0 and s.error == 0
    finally:
        dist.destroy_process_group()


def test_rank_step_refuses_wrong_gradient_copies():
    """RankStep hands the library raw addresses, so it checks the copies first: a copy of
    the wrong length or element size is refused before anything is enqueued."""
    import datetime
    import torch.distributed as dist

    import zero_partitioned_optimizer_shard_gb300 as z
    from zero_partitioned_optimizer_shard_gb300.ranks import RankStep, layout_for

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(_free_port())
    dist.init_process_group("gloo", rank=0, world_size=1, timeout=datetime.timedelta(seconds=30))
    try:
        lay = layout_for(100_000, 4)
        dev = torch.device("cuda", 0)
        rs = RankStep(lay, z.hparams(), z.ZERO_BF16, device=dev)
        P = lay.psi_padded
        good = [torch.zeros(P, dtype=torch.int16, device=dev) for _ in range(4)]
        for bad in ([torch.zeros(P - 8, dtype=torch.int16, device=dev)] + good[1:],
                    [torch.zeros(P, dtype=torch.float32, device=dev)] + good[1:],
                    good[:3]):
            with pytest.raises(ValueError):
                rs.step(bad)
        rs.step(good)  # all-zero gradients: a valid step
        s = z.zero_step_state_read(rs.st)
        assert s.t == 1 and s.norm == 0.0 and s.error == 0
    finally:
        dist.destroy_process_group()


def _full_main(proc, world, port, name, steps, starts, out_q):
    """The full-size workload's step on this process's ranks; returns, per step, the step
    state and the values at the sampled windows that fall in this process's range."""
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=proc, world_size=world)
    try:
        import zero_partitioned_optimizer_shard_gb300 as z
        from zero_partitioned_optimizer_shard_gb300.ranks import RankStep, layout_for

        wl = W.by_name(name)
        torch.cuda.set_device(0)
        dev = torch.device("cuda", 0)
        s = torch.cuda.current_stream(dev).cuda_stream
        lay = layout_for(wl.psi, wl.n_ranks, wl.stage, wl.bucket_elems)
        rs = RankStep(lay, z.hparams(**wl.hp.__dict__),
                      z.ZERO_F16 if wl.grad_dtype == "f16" else z.ZERO_BF16, wl.loss_scale,
                      wl.dynamic, wl.growth_interval, dev, exchange_elems=1 << 24)
        fills = [(rs.master, synth.ROLE_MASTER, synth.NORMAL, wl.master_sigma)]
        if wl.random_moments:
            fills += [(rs.m, synth.ROLE_MOM, synth.NORMAL, wl.mom_sigma),
                      (rs.v, synth.ROLE_VAR, synth.NORMAL_SQ, wl.mom_sigma)]
        for t_, role, kind, sig in fills:
            synth.fill_dev(t_.data_ptr(), synth.OUT_F32, kind, wl.state_key(role), rs.origin,
                           rs.local_len, wl.psi, sig, 1.0, s)
        mine = [b for b in starts if rs.origin <= b and b + 64 <= rs.origin + rs.local_len]
        flat = torch.tensor(np.concatenate([np.arange(b, b + 64) for b in mine]), device=dev)
        local = flat - rs.origin
        P = lay.psi_padded
        copies = [torch.empty(P, dtype=torch.int16, device=dev) for _ in range(rs.rank_count)]
        res = []
        for step in range(1, steps + 1):
            L = z.zero_step_state_read(rs.st).loss_scale
            for j, c in enumerate(copies):
                synth.fill_dev(c.data_ptr(), wl.grad_out, wl.grad_kind,
                               wl.grad_key(step, rs.rank_begin + j), 0, P, wl.psi, wl.grad_sigma,
                               L, s)
            inj = wl.injection(step)
            if inj and rs.rank_begin <= inj[0] < rs.rank_begin + rs.rank_count:
                copies[inj[0] - rs.rank_begin][inj[1]] = int(np.uint16(inj[2]).view(np.int16))
            rs.step(copies)
            st = z.zero_step_state_read(rs.st)
            vals = {k: getattr(rs, k).index_select(0, local).cpu().numpy()
                    for k in ("g", "master", "m", "v")}
            vals["out"] = rs.params.index_select(0, flat).cpu().numpy().view(np.uint16)
            res.append(((st.t, st.skip, st.norm, st.clip_coef, st.error, L, st.loss_scale),
                        mine, vals))
        out_q.put((proc, res))
    finally:
        dist.destroy_process_group()


def _full_size(name, world, steps, exchange_elems=1 << 24):
    from tests.golden import make_golden as golden
    from tests.gpu_harness import NORM_REL, bf16_ordinal
    from tests.test_gpu_fullsize import SampledOracle, _windows, WIN

    if not os.path.exists(golden.golden_path(name)):
        pytest.skip(f"golden file for {name} not generated")
    if torch.cuda.mem_get_info()[0] < 70e9:
        pytest.skip("needs ~60 GB of free HBM")
    wl = W.by_name(name)
    rows = golden.load(name)
    import oracle
    lay = oracle.load().partition(wl.psi, wl.n_ranks, wl.stage)
    starts = _windows(lay, wl)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_full_main, args=(p, world, port, name, steps, starts, q))
             for p in range(world)]
    for p in procs:
        p.start()
    got = {}
    try:
        for _ in range(world):
            r = q.get(timeout=1200)
            got[r[0]] = r[1]
    except queue.Empty:
        pytest.fail(f"processes {sorted(set(range(world)) - set(got))} returned nothing")
    finally:
        for p in procs:
            p.join(timeout=120)
            if p.is_alive():
                p.terminate()
    assert all(p.exitcode == 0 for p in procs)
    so = SampledOracle(wl, starts)
    skipped = 0
    for step in range(1, steps + 1):
        row = rows[step - 1]
        so.step(step, row)
        skipped += row["skipped"]
        want = {k: dict(zip(starts, getattr(so, k))) for k in ("g", "master", "m", "v", "out")}
        for p in range(world):
            (t, skip, norm, c, err, L, L_next), mine, vals = got[p][step - 1]
            assert err == 0 and (t, skip) == (row["t"], row["skipped"]), (p, step)
            assert (L, L_next) == (row["loss_scale"], row["loss_scale_next"]), (p, step)
            if not row["skipped"]:
                assert abs(norm - row["norm"]) <= NORM_REL * row["norm"], (p, step, norm)
                assert abs(c - row["clip_coef"]) <= 2 ** -23 * row["clip_coef"], (p, step)
            ga = vals["g"].reshape(len(mine), WIN)
            gb = np.stack([want["g"][s_] for s_ in mine])
            same = (ga.view(np.uint32) == gb.view(np.uint32)) | (np.isnan(ga) & np.isnan(gb))
            assert same.all(), (p, step, "g")
            for k in ("master", "m", "v"):
                a = vals[k].reshape(len(mine), WIN).astype(np.float64)
                b = np.stack([want[k][s_] for s_ in mine]).astype(np.float64)
                assert np.all(np.abs(a - b) <= 1e-5 * np.abs(b) + 1e-30), (p, step, k)
            o = vals["out"].reshape(len(mine), WIN)
            wo = np.stack([want["out"][s_] for s_ in mine])
            assert np.abs(bf16_ordinal(o) - bf16_ordinal(wo)).max() <= 1, (p, step)
    assert sum(len(got[p][0][1]) for p in range(world)) >= len(starts) - 2
    return skipped


def test_ranks_over_processes_full_size_gpt2():
    """The GPT-2-1.5B workload (psi = 1,557,611,200, N = 8) over two processes of four
    ranks, exchanging in 2^24-element windows: each step's norm, clip coefficient and t
    against the oracle's golden scalars, and the elements on sampled windows (every
    shard's start, middle and end, random places) against the oracle run on them."""
    _full_size("C2", 2, 2)


def test_ranks_over_processes_full_size_fp16_stress():
    """The fp16 dynamic-loss-scale stress workload (psi = 2^28, N = 16, Student-t
    gradients, L0 = 65536, an inf/NaN injected into rank 5's copy every 7th step) over two
    processes of eight ranks, 14 steps: the injections land in process 0's copies at
    flat indices of its own range, and natural fp16 overflows may land anywhere, so the
    skip decisions, the loss-scale sequence, t and the norms must agree with the golden
    oracle scalars step by step on both processes."""
    skipped = _full_size("C5", 2, 14)
    assert skipped >= 2


@pytest.mark.parametrize("psi,n,world,window", [
    (100_003, 4, 2, 0), (100_003, 4, 4, 8192), (48_761, 2, 2, 8192), (13, 4, 2, 0),
    ((1 << 20) + 77, 8, 4, 1 << 16), (3 * 8192 * 8 + 5, 8, 8, 8192),
])
def test_local_entry_points_write_only_their_buffers(psi, n, world, window):
    """The rank-local calls on guard-zoned buffers, the processes simulated one after the
    other in this process (the exchanges are plain copies): every local buffer's canary
    zones stay intact, and g, master, m, v and the gathered parameters equal the one-GPU
    step's bit for bit over two steps."""
    import zero_partitioned_optimizer_shard_gb300 as z
    from zero_partitioned_optimizer_shard_gb300.ranks import exchange_windows

    wl = replace(W.scaled(W.C2, psi, steps=2), n_ranks=n)
    ref = GpuRun(wl, split=True, align=8)
    lay, S, P = ref.lay, ref.lay.shard, ref.lay.psi_padded
    R = n // world
    L = R * S
    hp = ref.hp
    guard = GpuRun(wl, align=8)  # only its guarded allocator and canary check are used
    procs = []
    for p in range(world):
        loc = {k: guard.alloc(L, torch.float32) for k in ("g", "master", "m", "v")}
        for k in ("master", "m", "v"):
            loc[k].copy_(getattr(ref, k)[p * L:(p + 1) * L])
        loc["params"] = guard.alloc(P, torch.int16)
        loc["params"].zero_()
        loc["partials"] = guard.alloc(lay.n_tiles, torch.float64)
        loc["st"] = guard.alloc(z.STATE_BYTES, torch.uint8)
        loc["recv"] = [guard.alloc(L, torch.int16) for _ in range(n)]
        z.zero_step_state_init(lay, wl.loss_scale, wl.dynamic, wl.growth_interval, loc["st"],
                               loc["partials"])
        procs.append(loc)
    wins = exchange_windows(L, world, window)
    for step in (1, 2):
        ref.step(step)  # also leaves this step's gradient copies in ref.reps
        for p, loc in enumerate(procs):
            for k in range(n):  # every rank's copy of this process's range arrives
                loc["recv"][k].copy_(ref.reps[k][p * L:(p + 1) * L])
            for b, c in wins[p]:
                reps = [loc["recv"][k].data_ptr() + 2 * (b - p * L) for k in range(n)]
                z.zero_reduce_shard_unscale_local(lay, z.ZERO_BF16, p * R, R, reps, b, c,
                                                  loc["g"], loc["partials"], loc["st"])
        tpr = lay.tiles_per_rank
        flags = []
        for p, loc in enumerate(procs):  # the norm's inputs, exchanged
            for o, other in enumerate(procs):
                if o != p:
                    loc["partials"][o * R * tpr:(o + 1) * R * tpr] = \
                        other["partials"][o * R * tpr:(o + 1) * R * tpr]
            flags.append(int(loc["st"].view(torch.int32)[10]))
        for loc in procs:
            loc["st"].view(torch.int32)[10] = max(flags)
            z.zero_grad_norm(lay, hp, loc["partials"], loc["st"])
        for p, loc in enumerate(procs):
            z.zero_adamw_cast_gather_local(lay, hp, p * R, R, loc["g"], loc["master"], loc["m"],
                                           loc["v"], loc["params"][p * L:(p + 1) * L], loc["st"])
        for p, loc in enumerate(procs):  # the parameter all-gather
            for o, other in enumerate(procs):
                if o != p:
                    loc["params"][o * L:(o + 1) * L] = other["params"][o * L:(o + 1) * L]
        torch.cuda.synchronize()
        want = ref.arrays()
        for p, loc in enumerate(procs):
            sl = slice(p * L, (p + 1) * L)
            assert np.array_equal(loc["st"].cpu().numpy(), ref.st.cpu().numpy()), (step, p)
            for k in ("g", "master", "m", "v"):
                a = loc[k].cpu().numpy()
                assert np.array_equal(a.view(np.uint32), want[k][sl].view(np.uint32)), (step, p, k)
            assert np.array_equal(loc["params"].cpu().numpy().view(np.uint16), want["out"])
    guard.check_guards()
