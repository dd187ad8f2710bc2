"""GPU path vs the CPU oracle, element by element, through the C ABI (needs a GB300).

Sizes here are ones the oracle finishes in seconds while still spanning many 8192-element
tiles, shard boundaries in the middle of tiles and a padded ragged tail.  Expectations:
the reduced gradient g, indices, pads, flags, the skip decision and the loss-scale
sequence bit-exact; master/m/v within 1e-5 relative (and in practice bit-exact, since both
sides evaluate the same fp32 operations in the same order); the gathered bf16 parameters
within 1 ulp; the norm within 1e-5 relative.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import synth
import zero_partitioned_optimizer_shard_gb300 as z
from synth import workloads as W
from tests.gpu_harness import GpuRun, OracleRun, assert_scalars, assert_state_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _run_pair(wl, steps, bucket_elems=0, check_every=True):
    gpu = GpuRun(wl, bucket_elems)
    orc = OracleRun(wl)
    for s in range(1, steps + 1):
        st = gpu.step(s)
        rep = orc.step(s)
        assert_scalars(st, rep)
        if check_every or s == steps:
            exact = st.clip_coef == rep.clip_coef
            assert_state_close(gpu.arrays(), orc.arrays(), wl.psi, exact_expected=exact)
    gpu.check_guards()
    return gpu, orc


def test_c1_full_size():
    """C1 exactly: psi = 1,000,003 (odd; the last shard carries one pad), N = 4, fp16."""
    gpu, orc = _run_pair(W.C1, 1)
    s = gpu.state()
    assert s.t == 1 and s.skip == 0 and s.loss_scale == 1024.0 and s.n_steps == 1
    assert 0.45 < s.norm < 0.55 and s.clip_coef == 1.0  # clipping inactive in C1


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8, 16, 17, 33, 64])
def test_tiny_and_ragged(n):
    """Degenerate sizes: N > psi, one-element shards, shards of < 8 elements, 64 ranks."""
    for psi in (1, 2, 3, 7, 8, 9, 15, 16, 17, 31, 33, 63, 64, 65, 100, 257, 8195):
        dt = "f16" if (psi + n) % 2 else "bf16"
        wl = replace(W.scaled(W.C1, psi, steps=2), n_ranks=n, grad_dtype=dt,
                     loss_scale=1024.0 if dt == "f16" else 1.0, dynamic=dt == "f16",
                     random_moments=bool(psi % 3))
        _run_pair(wl, 2)


@pytest.mark.parametrize("recipe", ["C1", "C2"])
def test_fp16_gathered_parameters(recipe):
    """The fp16 variant of the gathered parameters (the FP16 replicated parameters of the
    ZeRO walkthrough's stage 1), for fp16 and bf16 gradients."""
    base = getattr(W, recipe)
    _run_pair(replace(W.scaled(base, 300_007, steps=2), hp=W.HP(params_dtype=z.ZERO_F16)), 2)


def test_tiles_shards_windows_bucketed_equals_whole():
    """Bucketed windows (tile pieces reduced in several launches) give the same bits."""
    psi = 4 * 3 * 8192 + 12345
    wl = replace(W.scaled(W.C2, psi, steps=2), n_ranks=4)
    ref, _ = _run_pair(wl, 2)
    want = ref.arrays()
    want_state = ref.state()
    for W_ in (8, 1000, 8192, 3 * 8192 + 8, psi // 3 // 8 * 8):
        got, _ = _run_pair(wl, 2, bucket_elems=W_, check_every=False)
        a = got.arrays()
        s = got.state()
        # tile pieces add up in another fp64 order: the norm may move in its last bits
        assert abs(s.norm - want_state.norm) <= 1e-13 * want_state.norm
        assert np.array_equal(a["g"].view(np.uint8), want["g"].view(np.uint8))
        if s.clip_coef == want_state.clip_coef:
            for k in want:
                assert np.array_equal(a[k].view(np.uint8), want[k].view(np.uint8)), (W_, k)


def test_reduce_windows_in_any_order():
    """The three entry points called directly, windows given out of order."""
    psi = 2 * 8192 * 5 + 77
    wl = replace(W.scaled(W.C2, psi, steps=1), n_ranks=5)
    gpu = GpuRun(wl)
    orc = OracleRun(wl)
    gpu.gen_grads(1)
    P = gpu.lay.psi_padded
    cuts = [0, 8, 8192, 20000, 20480, 40000, P]
    order = [3, 0, 5, 1, 4, 2]
    dt = z.ZERO_BF16
    for i in order:
        b, e = cuts[i], cuts[i + 1]
        reps = [r.data_ptr() + 2 * b for r in gpu.reps]
        z.zero_reduce_shard_unscale(gpu.lay, dt, reps, b, e - b, gpu.g, gpu.partials, gpu.st)
    z.zero_grad_norm(gpu.lay, gpu.hp, gpu.partials, gpu.st)
    z.zero_adamw_cast_gather(gpu.lay, gpu.hp, gpu.g, gpu.master, gpu.m, gpu.v, gpu.out, gpu.st)
    rep = orc.step(1)
    st = gpu.state()
    assert_scalars(st, rep)
    assert_state_close(gpu.arrays(), orc.arrays(), psi, exact_expected=st.clip_coef == rep.clip_coef)
    gpu.check_guards()


@pytest.mark.parametrize("bits", [0x7C00, 0x7E00, 0xFC00])
def test_overflow_skips_and_backs_off(bits):
    """A non-finite value in one rank's copy: flag set, step skipped, every state byte kept,
    L halved; the next step proceeds (fp16 dynamic scaling)."""
    wl = W.scaled(W.C1, 50_001, steps=3)
    gpu = GpuRun(wl)
    orc = OracleRun(wl)
    st = gpu.step(1)
    orc.step(1)
    before = gpu.arrays()
    L = gpu.gen_grads(2)
    gpu.reps[3][31337] = int(np.uint16(bits).view(np.int16))
    z.zero_step(gpu.lay, gpu.hp, z.ZERO_F16, gpu.bucket_ptrs(), gpu.g, gpu.partials, gpu.master,
                gpu.m, gpu.v, gpu.out, gpu.st)
    st = gpu.state()
    assert st.skip == 1 and st.t == 1 and st.loss_scale == L / 2 and st.n_skipped == 1
    assert st.overflow == 0  # cleared for the next step
    after = gpu.arrays()
    for k in ("master", "m", "v", "out"):
        assert np.array_equal(after[k].view(np.uint8), before[k].view(np.uint8)), k
    # the oracle, fed the same fault, agrees; then both run a clean step
    reps = orc.grads(2)
    reps[3][31337] = bits
    from oracle import F16
    rep = orc.orc.step(orc.lay, orc.hp, F16, reps, orc.g, orc.master, orc.m, orc.v, orc.out, orc.sc)
    assert rep.skipped == 1 and rep.loss_scale_next == st.loss_scale
    st = gpu.step(3)
    rep = orc.step(3)
    assert_scalars(st, rep)
    assert_state_close(gpu.arrays(), orc.arrays(), wl.psi, exact_expected=st.clip_coef == rep.clip_coef)
    gpu.check_guards()


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 values that are exact in bf16 -> their bf16 bit patterns."""
    u = np.asarray(x, np.float32).view(np.uint32)
    assert np.all(u & 0xFFFF == 0)
    return (u >> 16).astype(np.uint16)


@pytest.mark.parametrize("case", ["huge", "tiny", "mixed", "edge32"])
def test_sum_of_squares_at_the_range_edges(case):
    """Finite gradients far from 1: the per-tile sum of squares must not overflow or lose
    small terms.  'huge': three tiles of 2^60 (each tile's squares sum to 2^133, past the
    fp32 range; exact in fp64); 'tiny': magnitudes 2^-60 .. 2^-90 on both sides of the
    pair arithmetic's exact range; 'mixed': both kinds in one tile; 'edge32': a full tile
    just below the pair arithmetic's upper bound 2^32 (8192 squares summed in fp32 pairs
    reach 2^125 after the 2^24 scaling) and one at 2^33, just above it (fp64 path)."""
    psi, n = 5 * 8192 + 77, 4
    wl = W.scaled(W.C2, psi, steps=1)
    gpu = GpuRun(replace(wl, n_ranks=n))
    orc = OracleRun(replace(wl, n_ranks=n))
    P = gpu.lay.psi_padded
    rng = np.random.default_rng(17)
    vals = np.zeros((n, P), np.float32)
    if case in ("huge", "mixed"):
        vals[:, 1000:1000 + 3 * 8192] = np.float32(2.0 ** 60)
    if case == "edge32":
        vals[:, 8192:2 * 8192] = np.float32(1.9921875 * 2.0 ** 31)  # bf16-exact, < 2^32
        vals[:, 3 * 8192:4 * 8192] = np.float32(2.0 ** 33)
    if case in ("tiny", "mixed"):
        e = rng.integers(-90, -59, size=(n, psi))
        sgn = rng.choice([-1.0, 1.0], size=(n, psi))
        tiny = (sgn * np.ldexp(1.0, e)).astype(np.float32)
        sel = slice(0, psi) if case == "tiny" else slice(30000, psi)
        vals[:, sel] = tiny[:, sel]
    vals[:, psi:] = 0
    reps_np = [_bf16_bits(vals[k]) for k in range(n)]
    for k in range(n):
        gpu.reps[k].copy_(torch.from_numpy(reps_np[k].view(np.int16)))
    z.zero_step(gpu.lay, gpu.hp, z.ZERO_BF16, gpu.bucket_ptrs(), gpu.g, gpu.partials, gpu.master,
                gpu.m, gpu.v, gpu.out, gpu.st)
    st = gpu.state()
    from oracle import BF16
    rep = orc.orc.step(orc.lay, orc.hp, BF16, reps_np, orc.g, orc.master, orc.m, orc.v, orc.out,
                       orc.sc)
    assert np.isfinite(st.norm) and rep.norm > 0
    assert_scalars(st, rep)
    assert_state_close(gpu.arrays(), orc.arrays(), psi, exact_expected=st.clip_coef == rep.clip_coef)
    gpu.check_guards()


@pytest.mark.parametrize("n", [2, 8, 64])
def test_sharded_step_equals_unsharded_step(n):
    """The sharding identity of the ZeRO walkthrough (sec. 6(2): each rank updates its
    own partition, the all-gather reassembles [p0' ... p7']) on the GPU alone: N identical
    gradient copies average exactly to the copy, so the N-rank sharded step must equal
    the one-rank step on that copy bit for bit (clipping off, so no norm rounding enters;
    then with clipping on, within the norm's summation-order rounding)."""
    psi = 3 * 8192 + 1234
    for clip in (0.0, 1.0):
        hp = z.hparams(max_grad_norm=clip)
        runs = []
        for ranks in (n, 1):
            wl = replace(W.scaled(W.C2, psi, steps=2), n_ranks=ranks)
            gpu = GpuRun(wl, hp=hp)
            for step in (1, 2):
                gpu._fill(gpu.reps[0], wl.grad_out, wl.grad_kind, wl.grad_key(step, 0), wl.grad_sigma)
                for k in range(1, ranks):
                    gpu.reps[k].copy_(gpu.reps[0])
                z.zero_step(gpu.lay, gpu.hp, z.ZERO_BF16, gpu.bucket_ptrs(), gpu.g, gpu.partials,
                            gpu.master, gpu.m, gpu.v, gpu.out, gpu.st)
            gpu.check_guards()
            runs.append((gpu.state(), {k: v[:psi] for k, v in gpu.arrays().items()}))
        (sa, a), (sb, b) = runs
        assert sa.t == sb.t == 2
        if clip == 0.0:
            assert sa.clip_coef == sb.clip_coef == 1.0
            for k in a:
                assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), (n, k)
        else:
            assert abs(sa.norm - sb.norm) <= 1e-12 * sb.norm
            assert_state_close(dict(a, g=b["g"]), b, psi, exact_expected=sa.clip_coef == sb.clip_coef)


@pytest.mark.parametrize("recipe,psi,steps", [("C2", 2 * 3 * 4096 + 4097, 3),
                                              ("C2", 1_000_003, 2), ("C5", 200_003, 8)])
def test_rereading_schedule_equals_materialised_g(recipe, psi, steps):
    """zero_step with g = NULL at N = 2 (the reduce stores no g; AdamW re-reads the two
    gradient copies) gives the bits of the materialised-g step and the oracle's results;
    the fp16 recipe covers dynamic scaling, an injected overflow and fp16 parameters."""
    base = getattr(W, recipe)
    hp = W.HP(params_dtype=z.ZERO_F16) if recipe == "C5" else W.HP()
    wl = replace(W.scaled(base, psi, steps=steps), n_ranks=2, hp=hp, inject_rank=1)
    a, b = GpuRun(wl), GpuRun(wl)
    orc = OracleRun(wl)
    dt = z.ZERO_F16 if wl.grad_dtype == "f16" else z.ZERO_BF16
    for s in range(1, steps + 1):
        sa = a.step(s)
        b.gen_grads(s)
        z.zero_step(b.lay, b.hp, dt, b.bucket_ptrs(), None, b.partials, b.master, b.m, b.v, b.out,
                    b.st, b.stream)
        sb = b.state()
        rep = orc.step(s)
        assert (sa.skip, sa.t, sa.loss_scale, sa.clip_coef) == (sb.skip, sb.t, sb.loss_scale, sb.clip_coef)
        assert sa.norm == sb.norm or (sa.skip and sb.skip)
        assert_scalars(sb, rep)
        xa, xb = a.arrays(), b.arrays()
        for k in ("master", "m", "v", "out"):
            assert np.array_equal(xa[k].view(np.uint8), xb[k].view(np.uint8)), (s, k)
        want = orc.arrays()
        assert_state_close(dict(xb, g=want["g"]), want, wl.psi, exact_expected=sb.clip_coef == rep.clip_coef)
    a.check_guards()
    b.check_guards()


def test_bf16_static_scale_overflow_skips_without_backoff():
    wl = W.scaled(W.C2, 30_000, steps=1)
    gpu = GpuRun(wl)
    gpu.gen_grads(1)
    gpu.reps[0][12] = int(np.uint16(0x7F80).view(np.int16))  # bf16 +inf
    z.zero_step(gpu.lay, gpu.hp, z.ZERO_BF16, gpu.bucket_ptrs(), gpu.g, gpu.partials, gpu.master,
                gpu.m, gpu.v, gpu.out, gpu.st)
    st = gpu.state()
    assert st.skip == 1 and st.loss_scale == 1.0 and st.t == 0


def test_multistep_c2_recipe():
    """The GPT-2 workload's recipe (bf16, random state, clipping active) at 2^20+3, 10 steps."""
    _run_pair(W.scaled(W.C2, (1 << 20) + 3, steps=10), 10)


def test_c5_recipe_dynamic_scaling():
    """The fp16 stress recipe at psi = 2^20, N = 16, 50 steps: heavy tails, injected
    inf/NaN every 7th step, loss-scale back-off, clipping (threshold 0.2 here: the norm of
    this smaller buffer is about 0.45); flag and L bit-exact per step."""
    wl = replace(W.scaled(W.C5, 1 << 20, steps=50), hp=W.HP(max_grad_norm=0.2))
    gpu = GpuRun(wl)
    orc = OracleRun(wl)
    skipped = []
    for s in range(1, 51):
        st = gpu.step(s)
        rep = orc.step(s)
        assert_scalars(st, rep)
        skipped.append(rep.skipped)
        if s % 10 == 0 or rep.skipped:
            assert_state_close(gpu.arrays(), orc.arrays(), wl.psi,
                               exact_expected=st.clip_coef == rep.clip_coef)
    assert sum(skipped) >= 7 and all(skipped[s - 1] for s in range(7, 51, 7))
    gpu.check_guards()


def test_determinism_bitwise():
    wl = W.scaled(W.C2, 777_777, steps=2)
    results = []
    for _ in range(3):
        g = GpuRun(wl)
        g.step(1)
        s = g.step(2)
        a = g.arrays()
        results.append((s.norm, s.sumsq, {k: a[k].tobytes() for k in a}))
    for r in results[1:]:
        assert r[0] == results[0][0] and r[1] == results[0][1] and r[2] == results[0][2]


@pytest.mark.parametrize("wl", [W.scaled(W.C5, 200_000, steps=10),
                                replace(W.scaled(W.C2, 8 * 8192 * 200 + 5, steps=10), n_ranks=8)],
                         ids=["single-launch", "three-launch"])
def test_checkpoint_resume_bitwise(wl):
    """5 steps, save state + arrays, restore into fresh buffers, 5 more == 10 straight.  The
    saved state is written back with garbage in the kernels' internal counters, which
    zero_step_state_write must clear (the harness checks the chunk queue reads 0)."""
    a = GpuRun(wl)
    dt = z.ZERO_F16 if wl.grad_dtype == "f16" else z.ZERO_BF16
    assert (z.zero_step_launches(a.lay, dt) == 1) == (wl.psi < 1_000_000)
    for s in range(1, 11):
        a.step(s)
    b = GpuRun(wl)
    for s in range(1, 6):
        b.step(s)
    saved = b.state()
    arrs = {k: getattr(b, k).clone() for k in ("master", "m", "v", "out")}
    c = GpuRun(wl)
    for k, t in arrs.items():
        getattr(c, k).copy_(t)
    saved.arrivals, saved.launch_arrivals = 7, 9
    saved.adamw_next_chunk, saved.adamw_done = 12345, 3
    z.zero_step_state_write(c.st, saved)
    back = c.state()
    assert (back.arrivals, back.launch_arrivals) == (0, 0)
    for s in range(6, 11):
        c.step(s)
    x, y = a.arrays(), c.arrays()
    for k in ("master", "m", "v", "out"):
        assert np.array_equal(x[k].view(np.uint8), y[k].view(np.uint8)), k
    sa, sc = a.state(), c.state()
    assert (sa.t, sa.loss_scale, sa.norm, sa.n_steps) == (sc.t, sc.loss_scale, sc.norm, sc.n_steps)


@pytest.mark.parametrize("psi,n,stage", [(1 << 20, 2, 1), ((1 << 20) + 1, 64, 3), (1 << 22, 16, 2),
                                         ((1 << 22) + 1, 8, 1), (1 << 21, 4, 3),
                                         (3 * (1 << 20) + 5, 3, 2), ((1 << 21) + 7, 7, 2),
                                         ((1 << 21) + 3, 1, 2)])
def test_sweep_points_all_elements(psi, n, stage):
    """Bandwidth-sweep points (bf16 ~N(0,1e-3)) small enough for the oracle, every element."""
    _run_pair(W.sweep_point(psi, n, stage, steps=2), 2)


def test_stages_share_arithmetic():
    outs = []
    for stage in (1, 2, 3):
        g = GpuRun(W.sweep_point(100_003, 8, stage))
        g.step(1)
        outs.append(g.arrays())
    for o in outs[1:]:
        for k in o:
            assert np.array_equal(o[k].view(np.uint8), outs[0][k].view(np.uint8))


@pytest.mark.parametrize("recipe,steps,bucket,pinned", [("C2", 2, 65536, True), ("C5", 8, 65536, True),
                                                        ("C1", 3, 0, True), ("C1", 3, 0, False)])
def test_step_host_equals_device_path(recipe, steps, bucket, pinned):
    """zero_step_host (gradients in pinned host memory, bucketed H2D ring) gives the same
    bits as zero_step on device-resident gradients; with the fp16 dynamic-scale recipe
    the injected inf at step 7 is skipped the same way.  With one bucket of a small layout
    (the odd-size fp16 recipe) both take the single-launch step: it reads page-locked
    copies where they are (the staging buffer is left untouched), and pageable ones after
    they have been staged."""
    wl = W.scaled(getattr(W, recipe), 3 * 65536 + 40, steps=steps)
    dt = z.ZERO_F16 if wl.grad_dtype == "f16" else z.ZERO_BF16
    dev = GpuRun(wl, bucket_elems=bucket)
    host = GpuRun(wl, bucket_elems=bucket)
    P = host.lay.psi_padded
    if bucket == 0:
        assert z.zero_step_launches(host.lay, dt) == 1
    staging = torch.full((2 * wl.n_ranks * host.lay.bucket_elems,), 0x5A5A, dtype=torch.int16, device="cuda")
    copy_stream = torch.cuda.Stream()
    hstate = torch.empty(z.STATE_BYTES, dtype=torch.uint8).pin_memory()
    skipped = 0
    for s in range(1, steps + 1):
        dev.step(s)
        host.gen_grads(s)
        hreps = [r.cpu().pin_memory() if pinned else r.cpu() for r in host.reps]
        for r in host.reps:
            r.fill_(0x7F7F)  # the device copies must not be read
        z.zero_step_host(host.lay, host.hp, dt, hreps, staging, staging.numel() * 2,
                         host.g, host.partials, host.master, host.m, host.v, host.out, host.st,
                         hstate, None, copy_stream)
        torch.cuda.synchronize()
        hs = z.StepState.from_buffer_copy(hstate.numpy().tobytes())
        ds = dev.state()
        assert (hs.skip, hs.t, hs.loss_scale) == (ds.skip, ds.t, ds.loss_scale)
        assert hs.norm == ds.norm or (hs.skip and ds.skip)
        skipped += hs.skip
    assert hs.t == steps - skipped and skipped >= (1 if recipe == "C5" else 0)
    untouched = bool((staging == 0x5A5A).all())
    assert untouched == (bucket == 0 and pinned)  # read in place only on the single launch
    x, y = dev.arrays(), host.arrays()
    for k in x:
        assert np.array_equal(x[k].view(np.uint8), y[k].view(np.uint8)), k
    assert P == host.lay.psi_padded


@pytest.mark.parametrize("n,dtype,one_block", [(16, "bf16", False), (8, "bf16", True), (2, "f16", True)])
def test_step_host_reads_pinned_copies_in_place(n, dtype, one_block):
    """The single launch reading page-locked gradient copies in place, beyond the odd-size
    recipe: the N = 16 specialisation with bf16 copies, and copies that are views into ONE
    page-locked allocation (each copy's device address is an interior address of that
    one mapping, at the copy's offset).  Same bits as zero_step on device-resident copies
    over three steps, clipping active, and the staging buffer is never touched."""
    wl = replace(W.scaled(W.C2 if dtype == "bf16" else W.C1, (1 << 20) + 3, steps=3), n_ranks=n)
    dt = z.ZERO_F16 if dtype == "f16" else z.ZERO_BF16
    hp = z.hparams(max_grad_norm=1e-3)  # clipping active: c < 1 in every step
    dev = GpuRun(wl, hp=hp)
    host = GpuRun(wl, hp=hp)
    assert z.zero_step_launches(host.lay, dt) == 1
    P = host.lay.psi_padded
    slot = (host.lay.bucket_elems + 7) // 8 * 8
    staging = torch.full((2 * n * slot,), 0x5A5A, dtype=torch.int16, device="cuda")
    copy_stream = torch.cuda.Stream()
    hstate = torch.empty(z.STATE_BYTES, dtype=torch.uint8).pin_memory()
    stride = (P + 7) // 8 * 8 + 8  # copies 16-byte aligned, none at the allocation's start
    pool = torch.empty(n * stride + 8, dtype=torch.int16).pin_memory() if one_block else None
    for s in range(1, 4):
        dev.step(s)
        host.gen_grads(s)
        if one_block:  # copy k at element offset k * stride + 8
            hreps = [pool[k * stride + 8:k * stride + 8 + P] for k in range(n)]
            for h, r in zip(hreps, host.reps):
                h.copy_(r.cpu())
        else:
            hreps = [r.cpu().pin_memory() for r in host.reps]
        for r in host.reps:
            r.fill_(0x7F7F)  # the device copies must not be read
        z.zero_step_host(host.lay, host.hp, dt, hreps, staging, staging.numel() * 2,
                         host.g, host.partials, host.master, host.m, host.v, host.out, host.st,
                         hstate, None, copy_stream)
        torch.cuda.synchronize()
        hs = z.StepState.from_buffer_copy(hstate.numpy().tobytes())
        ds = dev.state()
        assert bytes(hs) == bytes(ds)
        assert hs.clip_coef < 1.0
    assert bool((staging == 0x5A5A).all())
    x, y = dev.arrays(), host.arrays()
    for k in x:
        assert np.array_equal(x[k].view(np.uint8), y[k].view(np.uint8)), k
    host.check_guards()


def test_device_rejects_bad_calls_without_side_effects():
    wl = W.scaled(W.C2, 10_000, steps=1)
    gpu = GpuRun(wl)
    gpu.step(1)
    before = gpu.arrays()
    with pytest.raises(z.ZeroError) as e:
        z.zero_reduce_shard_unscale(gpu.lay, z.ZERO_BF16, gpu.reps, 4, 8, gpu.g, gpu.partials, gpu.st)
    assert e.value.status == z.ZERO_EALIGN
    with pytest.raises(z.ZeroError):
        z.zero_adamw_cast_gather(gpu.lay, z.hparams(beta1=1.0), gpu.g, gpu.master, gpu.m, gpu.v,
                                 gpu.out, gpu.st)
    with pytest.raises(z.ZeroError):
        z.zero_step(gpu.lay, gpu.hp, z.ZERO_BF16, gpu.reps[:-1] + [0], gpu.g, gpu.partials,
                    gpu.master, gpu.m, gpu.v, gpu.out, gpu.st)
    after = gpu.arrays()
    for k in before:
        assert np.array_equal(after[k].view(np.uint8), before[k].view(np.uint8))
    gpu.check_guards()


def test_generator_twins_agree():
    """Device and host generators: same bits for every kind and output type (inputs)."""
    n = 1 << 20
    for out, kind, sigma, scale in [(synth.OUT_BF16, synth.NORMAL, 1e-4, 1.0),
                                    (synth.OUT_F16, synth.NORMAL, 1e-3, 1024.0),
                                    (synth.OUT_F16, synth.STUDENT_T3, 1e-3, 65536.0),
                                    (synth.OUT_F32, synth.NORMAL, 0.02, 1.0),
                                    (synth.OUT_F32, synth.NORMAL_SQ, 1e-4, 1.0)]:
        k = synth.key(7, 1, 3, 5)
        dt = torch.float32 if out == synth.OUT_F32 else torch.int16
        d = torch.empty(n, dtype=dt, device="cuda")
        begin = (1 << 33) + 12345  # a high flat offset exercises 64-bit counters
        synth.fill_dev(d.data_ptr(), out, kind, k, begin, n, begin + n - 100, sigma, scale)
        h = synth.fill_host(out, kind, k, begin, n, begin + n - 100, sigma, scale)
        assert np.array_equal(d.cpu().numpy().view(np.uint8), h.view(np.uint8))


@pytest.mark.parametrize("psi,launches", [(200_003, 1), (8 * 8192 * 60 + 3, 3)])
def test_zero_step_replays_from_a_cuda_graph(psi, launches):
    """zero_step enqueues kernels only (no host sync, no allocation), so a caller can
    capture it in a CUDA graph; replaying the graph gives the same bits as direct calls,
    for the single cooperative launch and for the three launches of a larger layout."""
    wl = W.scaled(W.C2, psi, steps=3)
    direct = GpuRun(wl)
    assert z.zero_step_launches(direct.lay, z.ZERO_BF16) == launches
    graphed = GpuRun(wl, guarded=False)
    stream = torch.cuda.Stream()
    graphed.stream = stream
    with torch.cuda.stream(stream):
        graphed.gen_grads(1)
        dt = z.ZERO_BF16
        ptrs = graphed.bucket_ptrs()
        # first call outside the capture (per-device set-up: occupancy, shared-memory size)
        z.zero_step(graphed.lay, graphed.hp, dt, ptrs, graphed.g, graphed.partials, graphed.master,
                    graphed.m, graphed.v, graphed.out, graphed.st, stream)
        direct.step(1)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            z.zero_step(graphed.lay, graphed.hp, dt, ptrs, graphed.g, graphed.partials,
                        graphed.master, graphed.m, graphed.v, graphed.out, graphed.st, stream)
        for s in (2, 3):
            graphed.gen_grads(s)
            g.replay()
            direct.step(s)
        torch.cuda.synchronize()
    a, b = direct.arrays(), graphed.arrays()
    for k in a:
        assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k
    sa, sb = direct.state(), graphed.state()
    assert (sa.t, sa.norm, sa.clip_coef) == (sb.t, sb.norm, sb.clip_coef) and sa.t == 3


def test_buckets_reduced_while_a_producer_writes_the_next():
    """Gradient buckets produced on one stream and reduced on another through a two-slot
    ring of constant-size buffers give the same bits as one zero_step on all copies, and
    the oracle's step within the stated tolerances, after every step."""
    wl = W.scaled(W.C3, 5 * 65536 + 1000, steps=2)
    Wb = 65536
    ref = GpuRun(wl, bucket_elems=Wb)
    pipe = GpuRun(wl, bucket_elems=Wb, guarded=False)
    orc = OracleRun(wl)
    lay, N, P = pipe.lay, pipe.lay.n_ranks, pipe.lay.psi_padded
    comp = pipe.stream
    prod = torch.cuda.Stream()
    ring = [[torch.empty(Wb, dtype=torch.int16, device="cuda") for _ in range(N)] for _ in range(2)]
    filled = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    for step in (1, 2):
        ref.step(step)
        prod.wait_stream(comp)
        for b in range(lay.n_buckets):
            slot, begin = b & 1, b * Wb
            count = min(Wb, P - begin)
            if b >= 2:
                prod.wait_event(consumed[slot])
            for k in range(N):
                synth.fill_dev(ring[slot][k].data_ptr(), wl.grad_out, wl.grad_kind,
                               wl.grad_key(step, k), begin, count, wl.psi, wl.grad_sigma, 1.0,
                               prod.cuda_stream)
            filled[slot].record(prod)
            comp.wait_event(filled[slot])
            z.zero_reduce_shard_unscale(lay, z.ZERO_BF16, [r.data_ptr() for r in ring[slot]], begin,
                                        count, pipe.g, pipe.partials, pipe.st, comp)
            consumed[slot].record(comp)
        z.zero_grad_norm(lay, pipe.hp, pipe.partials, pipe.st, comp)
        z.zero_adamw_cast_gather(lay, pipe.hp, pipe.g, pipe.master, pipe.m, pipe.v, pipe.out, pipe.st,
                                 comp)
        assert_scalars(pipe.state(), orc.step(step))
        assert_state_close(pipe.arrays(), orc.arrays(), wl.psi, exact_expected=False)
    torch.cuda.synchronize()
    a, b = ref.arrays(), pipe.arrays()
    for k in a:
        assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k
