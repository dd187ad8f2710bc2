"""A checked build of the library: every store of the reduce pass and of the single-launch
step first checks that it lies in the range the storing block owns (its tile of the flat
buffer, its shared-memory arrays); a failed check records 2 in the step state's error word
and skips the store.  The test builds that variant (-DZERO_CHECKED; the product library has
no checks and no such switch), runs steps through it on ragged layouts of every shape
(single launch staged and unstaged, three launches, bucketed windows, g = NULL), and
requires error word 0 and the product library's bits.  Out-of-range writes inside a
buffer, which canary zones cannot see, would show up here."""
import ctypes as C
import os
import subprocess
from dataclasses import replace

import numpy as np
import pytest
import torch

import zero_partitioned_optimizer_shard_gb300 as z
from synth import workloads as W
from tests.gpu_harness import GpuRun
from zero_partitioned_optimizer_shard_gb300 import _build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked(tmp_path_factory):
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()
    d = tmp_path_factory.mktemp("checked")
    objs, procs = [], []
    for src in _build.SOURCES:
        o = str(d / (os.path.splitext(src)[0] + ".o"))
        procs.append(subprocess.Popen(["nvcc", *_build.NVCC_FLAGS, "-DZERO_CHECKED", "-c",
                                       os.path.join(_build.CSRC, src), "-o", o]))
        objs.append(o)
    assert all(p.wait() == 0 for p in procs)
    lib = str(d / "libzero_shard_checked.so")
    arch = _build.ARCH
    subprocess.run(["nvcc", "-shared", f"-gencode=arch=compute_{arch},code=sm_{arch}", "-o", lib,
                    *objs, "-lcudart"], check=True)
    product = z.lib()
    saved_path = z.LIB_PATH
    z.LIB_PATH, z._L = lib, None
    handle = z.lib()  # the checked library, with the binding's argument types
    z.LIB_PATH, z._L = saved_path, product
    yield handle
    z._L = product


class _Using:
    """Route the binding's calls to another library handle for the duration of a block."""

    def __init__(self, handle):
        self.handle = handle

    def __enter__(self):
        self.saved, z._L = z._L, self.handle

    def __exit__(self, *exc):
        z._L = self.saved


CASES = [
    # (workload, bucket elements)
    (W.C1, 0),                                                        # single launch, staged
    (W.scaled(W.C2, 8 * 8192 * 20 + 5, steps=2), 0),                  # single launch, unstaged
    (replace(W.scaled(W.C2, 64 * 9000 + 3, steps=2), n_ranks=64), 0),  # generic, unstaged
    (W.scaled(W.C2, (1 << 24) + 3, steps=2), 0),                      # three launches
    (W.scaled(W.C3, 5 * 65536 + 1000, steps=2), 65536),               # bucketed windows
] + [(replace(W.scaled(W.C1, psi, steps=2), n_ranks=n), 0)
     for n in (1, 3, 8, 17, 64) for psi in (1, 7, 33, 65, 257, 8195)]


@pytest.mark.parametrize("wl,bucket", CASES, ids=lambda v: getattr(v, "name", str(v)))
def test_checked_build_owns_every_store(checked, wl, bucket):
    ref = GpuRun(wl, bucket)
    chk = GpuRun(wl, bucket)
    for step in range(1, min(wl.steps, 2) + 1):
        ref.step(step)
        with _Using(checked):
            chk.step(step)
        s = chk.state()
        assert s.error == 0, f"a store outside its block's range (error word {s.error})"
        assert bytes(s) == bytes(ref.state())
        a, b = chk.arrays(), ref.arrays()
        for k in a:
            assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k
    chk.check_guards()


def test_checked_build_without_g(checked):
    """N = 2, g = NULL (the re-reading schedule on three launches, nothing on one)."""
    for psi in (2 * 8192 * 7 + 3, (1 << 22) + 9):
        wl = replace(W.scaled(W.C2, psi, steps=2), n_ranks=2)
        gpu = GpuRun(wl)
        gpu.gen_grads(1)
        with _Using(checked):
            z.zero_step(gpu.lay, gpu.hp, z.ZERO_BF16, gpu.bucket_ptrs(), None, gpu.partials,
                        gpu.master, gpu.m, gpu.v, gpu.out, gpu.st, gpu.stream)
        assert gpu.state().error == 0
        gpu.check_guards()
