"""The single-launch step that zero_step takes for small layouts (k_step_fused), in both
of its shapes: staged (at most one tile per SM; the tile's optimizer state is copied into
shared memory) and unstaged (more tiles than SMs).

It must give the same bits as the three separate calls (reduce, norm, AdamW) in every
output and in the whole 128-byte step state, over several steps, on ragged sizes, every
specialised and generic rank count, fp16 and bf16 gradients, fp16 gathered parameters,
an injected overflow (skipped step, scale back-off) and the degenerate sizes; it must
match the oracle; and zero_step_launches must say which path a layout takes.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import zero_partitioned_optimizer_shard_gb300 as z
from synth import workloads as W
from tests.gpu_harness import GpuRun, OracleRun, assert_scalars, assert_state_close, dtype_code

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


CASES = {
    # the odd-size fp16 workload at its full size: 1,000,003 parameters, N = 4
    "c1": replace(W.C1, steps=2),
    # generic kernel (N = 3), shards not a multiple of the tile, ragged end
    "n3-ragged": replace(W.scaled(W.C2, 3 * 8192 * 5 + 77, steps=3), n_ranks=3),
    "n2": replace(W.scaled(W.C2, 2 * 8192 * 9 + 13, steps=3), n_ranks=2),
    "n8": W.scaled(W.C2, 8 * 8192 * 6 + 5, steps=3),
    # fp16 dynamic scale, Student-t gradients, +inf injected into rank 5 at step 7
    "n16-overflow": W.scaled(W.C5, 16 * 8192 * 3 + 9, steps=8),
    "n64": replace(W.scaled(W.C2, 64 * 9000 + 3, steps=2), n_ranks=64),
    "fp16-params": replace(W.scaled(W.C2, 4 * 8192 * 4 + 1, steps=2), n_ranks=4,
                           hp=replace(W.C2.hp, params_dtype=z.ZERO_F16)),
    "no-clip": replace(W.scaled(W.C2, 8 * 5000 + 1, steps=2),
                       hp=replace(W.C2.hp, max_grad_norm=0.0)),
    # clipping active in every step (c < 1): the staged shape's speculative update with
    # c = 1 is dropped and the tile is updated again from its shared-memory copies
    "clip-active": replace(W.scaled(W.C2, 8 * 8192 * 4 + 3, steps=3),
                           hp=replace(W.C2.hp, max_grad_norm=1e-4)),
    "psi5": replace(W.scaled(W.C1, 5, steps=2), n_ranks=4),
    "psi1": replace(W.scaled(W.C1, 1, steps=2), n_ranks=4),
    # more tiles than SMs: the unstaged shape (up to 3 blocks per SM, state read from L2)
    "n8-many-tiles": W.scaled(W.C2, 8 * 8192 * 20 + 5, steps=2),
    "n3-many-tiles": replace(W.scaled(W.C2, 3 * 8192 * 60 + 1, steps=2), n_ranks=3),
}


@pytest.mark.parametrize("ulps", [-2, 0, 1, 40])
def test_clip_threshold_same_bits_as_split(ulps):
    """max_grad_norm a few float ulps around norm + 1e-6, so c is 1 exactly or just below.
    Close to that threshold the single launch cannot release its blocks on the fp32
    upper bound of the sum of squares and forms the exact norm first (ulps -2, 0, 1);
    further above it releases them on the bound (40).  Both must give the separate
    calls' bits."""
    base = W.scaled(W.C2, 8 * 8192 * 4 + 3, steps=1)
    norm = GpuRun(base).step(1).norm
    m = np.float32(norm + 1e-6)
    if float(m) < norm + 1e-6:
        m = np.nextafter(m, np.float32(np.inf))  # the least float >= norm + 1e-6
    for _ in range(abs(ulps)):
        m = np.nextafter(m, np.float32(np.inf if ulps > 0 else -np.inf))
    wl = replace(base, hp=replace(base.hp, max_grad_norm=float(m)))
    fused, split = GpuRun(wl), GpuRun(wl, split=True)
    assert z.zero_step_launches(fused.lay, dtype_code(wl)) == 1
    sf, ss = fused.step(1), split.step(1)
    assert bytes(sf) == bytes(ss), (sf.clip_coef, ss.clip_coef)
    _arrays_equal(fused.arrays(), split.arrays())
    if ulps >= 1:
        assert sf.clip_coef == 1.0
    if ulps < 0:
        assert sf.clip_coef < 1.0


def _arrays_equal(a: dict, b: dict):
    for k in a:
        assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k


@pytest.mark.parametrize("name", list(CASES))
def test_single_launch_equals_split_calls_bit_for_bit(name):
    wl = CASES[name]
    fused = GpuRun(wl)
    split = GpuRun(wl, split=True)
    assert z.zero_step_launches(fused.lay, dtype_code(wl)) == 1
    skipped = 0
    for step in range(1, wl.steps + 1):
        sf, ss = fused.step(step), split.step(step)
        assert bytes(sf) == bytes(ss), (step, sf.norm, ss.norm, sf.clip_coef, ss.clip_coef)
        assert sf.error == 0 and sf.arrivals == 0 and sf.launch_arrivals == 0
        assert sf.applied_c == (-1.0 if sf.skip else sf.clip_coef)
        if name == "clip-active":
            assert sf.clip_coef < 1.0
        skipped += sf.skip
        _arrays_equal(fused.arrays(), split.arrays())
    if wl.inject_every:
        assert skipped >= 1
    fused.check_guards()
    split.check_guards()


@pytest.mark.parametrize("name", ["c1", "n16-overflow", "n3-ragged", "clip-active"])
def test_single_launch_matches_oracle(name):
    wl = CASES[name]
    gpu = GpuRun(wl)
    orc = OracleRun(wl)
    assert z.zero_step_launches(gpu.lay, dtype_code(wl)) == 1
    for step in range(1, wl.steps + 1):
        s = gpu.step(step)
        rep = orc.step(step)
        assert_scalars(s, rep)
        assert_state_close(gpu.arrays(), orc.arrays(), wl.psi,
                           exact_expected=bool(rep.skipped) or s.clip_coef == rep.clip_coef)
    gpu.check_guards()


def test_both_shapes_are_exercised():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = [z.zero_partition(w.psi, w.n_ranks, w.stage).n_tiles for w in CASES.values()]
    assert min(tiles) <= sms < max(tiles)


def test_launch_counts():
    bf = z.ZERO_BF16
    assert z.zero_step_launches(z.zero_partition(1_000_003, 4, 2), z.ZERO_F16) == 1
    # more than 128 tile slots per rank: the three-launch step
    lay = z.zero_partition(1 << 24, 4, 2)
    assert lay.tiles_per_rank > 128 and z.zero_step_launches(lay, bf) == 3
    # bucketed: a reduce launch per bucket
    lay = z.zero_partition(300_000, 4, 2, 1, 65536)
    assert z.zero_step_launches(lay, bf) == lay.n_buckets + 2
    # more tiles than can be resident at once (3 blocks per SM at most)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    lay = z.zero_partition(64 * 8192 * 100, 64, 2)
    assert lay.n_tiles > 4 * sms and z.zero_step_launches(lay, bf) == 3


def test_single_launch_without_g_equals_with_g():
    """N = 2 with g = NULL: nothing but g differs (it is not written)."""
    wl = replace(W.scaled(W.C2, 2 * 8192 * 7 + 3, steps=3), n_ranks=2)
    with_g = GpuRun(wl)
    no_g = GpuRun(wl)
    no_g.g.fill_(7.0)
    dt = dtype_code(wl)
    for step in range(1, wl.steps + 1):
        with_g.step(step)
        no_g.gen_grads(step)
        z.zero_step(no_g.lay, no_g.hp, dt, no_g.bucket_ptrs(), None, no_g.partials, no_g.master,
                    no_g.m, no_g.v, no_g.out, no_g.st, no_g.stream)
        assert bytes(with_g.state()) == bytes(no_g.state())
    a, b = with_g.arrays(), no_g.arrays()
    for k in ("master", "m", "v", "out"):
        assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k
    assert np.all(b["g"] == 7.0)  # never written
    no_g.check_guards()


def test_split_calls_after_single_launch_steps():
    """The partials and the arrival counter are left as the split calls expect them:
    single-launch steps and split steps may alternate on one state."""
    wl = W.scaled(W.C2, 8 * 8192 * 3 + 11, steps=4)
    mixed = GpuRun(wl)
    split = GpuRun(wl, split=True)
    for step in range(1, 5):
        mixed.split = step % 2 == 0
        assert bytes(mixed.step(step)) == bytes(split.step(step))
    _arrays_equal(mixed.arrays(), split.arrays())
    assert float(mixed.partials.abs().sum()) == 0.0
