"""A device wait that runs out reports an error status and leaves the GPU usable.

k_adamw waits on mbarriers for its bulk copies, and the single-launch step's blocks wait
for the block that forms the norm; every such wait is bounded (~2 s).
To exercise the timeout path without any fault, the test builds a test-only variant of
the library (-DZERO_TEST_HOOKS; the product library has no such switch) in which one
chunk's barrier is armed but its copies are withheld: a flag that nothing sets.  The
kernel must give up, record 1 in the step state's error word, wait (bounded) for its
other copies in flight and leave; the host sees a normal completion and reads the
status; and the same process then runs a full step through the product library that
still matches the oracle.
"""
import ctypes as C
import time

import numpy as np
import pytest
import torch

import zero_partitioned_optimizer_shard_gb300 as z
from synth import workloads as W
from tests.gpu_harness import GpuRun, OracleRun, assert_scalars, assert_state_close

pytestmark = pytest.mark.gpu


def test_adamw_wait_runs_out_reports_error_and_gpu_stays_usable(hooked):
    # 3 chunks of 4096 elements per block on average (the blocks take them from a queue)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    wl = W.scaled(W.C2, sms * 4096 * 3 + 123, steps=1)
    gpu = GpuRun(wl, guarded=False)
    gpu.gen_grads(1)
    dt = z.ZERO_BF16
    z.zero_reduce_shard_unscale(gpu.lay, dt, gpu.reps, 0, gpu.lay.psi_padded, gpu.g, gpu.partials,
                                gpu.st)
    z.zero_grad_norm(gpu.lay, gpu.hp, gpu.partials, gpu.st)
    assert gpu.state().error == 0
    assert hooked.zero_test_withhold_adamw_chunk(sms + 5) == 0  # whichever block takes it
    t0 = time.time()
    rc = hooked.zero_adamw_cast_gather(C.byref(gpu.lay), C.byref(gpu.hp), gpu.g.data_ptr(),
                                       gpu.master.data_ptr(), gpu.m.data_ptr(), gpu.v.data_ptr(),
                                       gpu.out.data_ptr(), gpu.st.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()  # completes: the wait gave up, no fault
    waited = time.time() - t0
    assert hooked.zero_test_withhold_adamw_chunk(~0 & 0xFFFFFFFFFFFFFFFF) == 0
    s = gpu.state()
    assert s.error == 1, s.error
    assert 1.0 < waited < 60.0, waited
    # the block that gave up still counted itself done, so the last block put the chunk
    # queue back to 0 for the next launch
    assert (s.adamw_next_chunk, s.adamw_done) == (0, 0), (s.adamw_next_chunk, s.adamw_done)
    # the context is still good: a full step through the product library matches the oracle
    wl2 = W.scaled(W.C2, 300_007, steps=1)
    fresh = GpuRun(wl2)
    orc = OracleRun(wl2)
    st = fresh.step(1)
    rep = orc.step(1)
    assert st.error == 0
    assert_scalars(st, rep)
    assert_state_close(fresh.arrays(), orc.arrays(), wl2.psi, exact_expected=st.clip_coef == rep.clip_coef)
    fresh.check_guards()


def test_single_launch_wait_runs_out_reports_error_and_gpu_stays_usable(hooked):
    """The single-launch step's blocks wait for the last block to form the norm; with one
    block absent (test build only) that wait runs out after ~2 s: the error word reads 1,
    no parameter or optimizer-state byte is written, and the GPU stays usable."""
    hooked.zero_test_absent_fused_block.argtypes = [C.c_ulonglong]
    hooked.zero_test_absent_fused_block.restype = C.c_int
    hooked.zero_step.argtypes = [C.POINTER(z.Layout), C.POINTER(z.HParams), C.c_int,
                                 C.POINTER(C.c_void_p)] + [C.c_void_p] * 8
    hooked.zero_step.restype = C.c_int
    wl = W.scaled(W.C2, 8 * 8192 * 4 + 17, steps=1)
    gpu = GpuRun(wl, guarded=False)
    assert z.zero_step_launches(gpu.lay, z.ZERO_BF16) == 1
    gpu.gen_grads(1)
    before = gpu.arrays()
    assert hooked.zero_test_absent_fused_block(3) == 0
    ptrs = (C.c_void_p * len(gpu.reps))(*[r.data_ptr() for r in gpu.reps])
    t0 = time.time()
    rc = hooked.zero_step(C.byref(gpu.lay), C.byref(gpu.hp), z.ZERO_BF16, ptrs, gpu.g.data_ptr(),
                          gpu.partials.data_ptr(), gpu.master.data_ptr(), gpu.m.data_ptr(),
                          gpu.v.data_ptr(), gpu.out.data_ptr(), gpu.st.data_ptr(),
                          torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()  # completes: every wait gave up, no fault
    waited = time.time() - t0
    assert hooked.zero_test_absent_fused_block(~0 & 0xFFFFFFFFFFFFFFFF) == 0
    s = gpu.state()
    assert s.error == 1 and s.t == 0, (s.error, s.t)
    assert 1.0 < waited < 60.0, waited
    after = gpu.arrays()
    for k in ("master", "m", "v", "out"):
        assert np.array_equal(before[k].view(np.uint8), after[k].view(np.uint8)), k
    # the context is still good: a full step through the product library matches the oracle
    wl2 = W.scaled(W.C2, 300_007, steps=1)
    fresh = GpuRun(wl2)
    orc = OracleRun(wl2)
    st = fresh.step(1)
    rep = orc.step(1)
    assert st.error == 0
    assert_scalars(st, rep)
    assert_state_close(fresh.arrays(), orc.arrays(), wl2.psi, exact_expected=st.clip_coef == rep.clip_coef)
    fresh.check_guards()
