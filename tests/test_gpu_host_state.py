"""Optimizer state offloaded to host memory: zero_adamw_cast_gather_host_state (needs a GB300).

master, m and v live in page-locked host memory and the kernel updates them in place
over the CPU-GPU link.  The arithmetic is the device path's, so the results must be the
oracle's (same expectations as the device-resident parity tests) and bit-identical to the
device-resident path.  Host buffers sit between canary zones like the device ones.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import zero_partitioned_optimizer_shard_gb300 as z
from synth import workloads as W
from tests.gpu_harness import GpuRun, OracleRun, assert_scalars, assert_state_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()


def _run_pair(wl, steps, bucket_elems=0):
    gpu = GpuRun(wl, bucket_elems, host_state=True)
    assert not gpu.master.is_cuda and gpu.master.is_pinned()
    orc = OracleRun(wl)
    for s in range(1, steps + 1):
        st = gpu.step(s)
        rep = orc.step(s)
        assert_scalars(st, rep)
        assert_state_close(gpu.arrays(), orc.arrays(), wl.psi,
                           exact_expected=st.clip_coef == rep.clip_coef)
    gpu.check_guards()
    return gpu


@pytest.mark.parametrize("psi", [1, 7, 4097, 1_000_003])
def test_host_state_matches_oracle(psi):
    """GPT-2 recipe (bf16 copies, random moments, clipping active), ragged sizes."""
    _run_pair(W.scaled(W.C2, psi, steps=3), 3)


def test_host_state_fp16_dynamic_scale_and_skip():
    """C5 recipe (fp16, Student-t, injected inf/NaN at step 7): the skipped step leaves the
    host-resident state byte-identical; fp16 gathered parameters."""
    wl = replace(W.scaled(W.C5, 200_003, steps=8), hp=W.HP(params_dtype=z.ZERO_F16))
    gpu = _run_pair(wl, 6)
    before = gpu.arrays()
    st = gpu.step(7)
    assert st.skip == 1
    after = gpu.arrays()
    for k in ("master", "m", "v", "out"):
        assert np.array_equal(after[k].view(np.uint8), before[k].view(np.uint8)), k


def test_host_state_bucketed_windows():
    wl = replace(W.scaled(W.C2, 3 * 65536 + 1001, steps=2), n_ranks=5)
    _run_pair(wl, 2, bucket_elems=65536)


def test_host_state_bits_equal_device_state():
    wl = W.scaled(W.C2, 2_000_001, steps=2)
    dev = GpuRun(wl)
    host = GpuRun(wl, host_state=True)
    for s in (1, 2):
        a, b = dev.step(s), host.step(s)
        assert (a.norm, a.clip_coef, a.t) == (b.norm, b.clip_coef, b.t)
    x, y = dev.arrays(), host.arrays()
    for k in x:
        assert np.array_equal(x[k].view(np.uint8), y[k].view(np.uint8)), k
    dev.check_guards()
    host.check_guards()


def test_host_state_rejects_device_and_pageable_memory():
    wl = W.scaled(W.C2, 10_000, steps=1)
    gpu = GpuRun(wl, host_state=True)
    gpu.step(1)
    before = gpu.arrays()
    P = gpu.lay.psi_padded
    on_device = torch.zeros(P, dtype=torch.float32, device="cuda:0")
    pageable = torch.zeros(P, dtype=torch.float32)
    assert not pageable.is_pinned()
    for bad in ((on_device, gpu.m, gpu.v), (gpu.master, pageable, gpu.v),
                (gpu.master, gpu.m, on_device)):
        with pytest.raises(z.ZeroError) as e:
            z.zero_adamw_cast_gather_host_state(gpu.lay, gpu.hp, gpu.g, *bad, gpu.out, gpu.st)
        assert e.value.status == z.ZERO_EINVAL
    after = gpu.arrays()
    for k in before:
        assert np.array_equal(after[k].view(np.uint8), before[k].view(np.uint8)), k
    gpu.check_guards()
