"""zero_step_static_workspace: the step for callers that cannot allocate device memory.

Such a caller cannot give the library a scratch buffer (its memory manager already holds
the GPU's memory, or it must not take the synchronisation a cudaMalloc/cudaFree can
cause mid-step), so this entry point keeps the per-tile sum-of-squares partials in a
static device array inside the library.  The test calls it through the C ABI twice in a
row and checks every output against zero_step, the entry point with a caller-provided
workspace, on identical inputs, within the tolerances the other GPU tests use; around the
second call it checks that neither torch's allocator nor the device's free memory moved.  It
passes alone in a fresh process and after the rest of the suite (the array keeps the
previous call's contents, and each call clears the slots it uses).
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import zero_partitioned_optimizer_shard_gb300 as z
from synth import workloads as W
from tests.gpu_harness import GpuRun, NORM_REL, REL, FLOOR, bf16_ordinal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _close(a: dict, b: dict, psi: int):
    ga, gb = a["g"], b["g"]
    assert np.array_equal(ga.view(np.uint32), gb.view(np.uint32))
    for k in ("master", "m", "v"):
        x, y = a[k].astype(np.float64), b[k].astype(np.float64)
        assert np.all(np.abs(x - y) <= REL * np.abs(y) + FLOOR), k
        assert np.array_equal(a[k][psi:].view(np.uint32), b[k][psi:].view(np.uint32))
    assert np.abs(bf16_ordinal(a["out"]) - bf16_ordinal(b["out"])).max() <= 1


@pytest.mark.parametrize("wl,bucket", [
    (replace(W.scaled(W.C2, 5 * 8192 * 8 + 123, steps=2), n_ranks=8), 0),
    (W.scaled(W.C1, 300_007, steps=2), 65536),
])
def test_static_workspace_matches_zero_step_twice(wl, bucket):
    ref = GpuRun(wl, bucket)
    new = GpuRun(wl, bucket)
    # initialise the second run's state without a separate workspace: g stands in
    z.zero_step_state_init(new.lay, wl.loss_scale, wl.dynamic, wl.growth_interval, new.st, new.g)
    dt = z.ZERO_F16 if wl.grad_dtype == "f16" else z.ZERO_BF16
    for step in (1, 2):
        ref.step(step)
        new.gen_grads(step)
        torch.cuda.synchronize()
        before = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
        z.zero_step_static_workspace(new.lay, new.hp, dt, new.bucket_ptrs(), new.g, new.master,
                                     new.m, new.v, new.out, new.st)
        torch.cuda.synchronize()
        after = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
        if step > 1:
            # the first call on the device may load the library's kernels (lazy module
            # loading); every later call must leave the device's free memory as it was
            assert after == before, f"device memory changed across the call: {before} -> {after}"
        sr, sn = ref.state(), new.state()
        assert (sn.t, sn.skip, sn.loss_scale, sn.n_steps) == (sr.t, sr.skip, sr.loss_scale, sr.n_steps)
        assert abs(sn.norm - sr.norm) <= NORM_REL * sr.norm
        assert sn.clip_coef == sr.clip_coef
        _close(new.arrays(), ref.arrays(), wl.psi)
    new.check_guards()


def test_static_workspace_rejects_oversized_layout():
    # 9e9 parameters over 64 ranks: 64 * (ceil(140,625,000 / 8192) + 1) = 1,098,752 tiles,
    # more than the array's 2^20 slots; rejected on the host before anything is enqueued
    lay = z.zero_partition(9_000_000_000, 64, 2)
    assert lay.n_tiles == 1_098_752 > (1 << 20)
    with pytest.raises(z.ZeroError) as e:
        z.zero_step_static_workspace(lay, z.hparams(), z.ZERO_BF16, [16] * 64, 16, 16, 16, 16, 16, 16)
    assert e.value.status == z.ZERO_ENOMEM
