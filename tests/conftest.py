import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running")


@pytest.fixture(scope="session")
def hooked(tmp_path_factory):
    """The library built with -DZERO_TEST_HOOKS (test-only entry points; the product library
    has no such switch), as a ctypes handle.  Built once per session, on a GPU machine."""
    import ctypes as C
    import subprocess

    import torch

    import __graft_entry__
    import zero_partitioned_optimizer_shard_gb300 as z
    from zero_partitioned_optimizer_shard_gb300 import _build

    __graft_entry__.build()
    assert torch.cuda.is_available()
    d = tmp_path_factory.mktemp("hooked")
    objs, procs = [], []
    for src in _build.SOURCES:
        o = str(d / (os.path.splitext(src)[0] + ".o"))
        procs.append(subprocess.Popen(["nvcc", *_build.NVCC_FLAGS, "-DZERO_TEST_HOOKS", "-c",
                                       os.path.join(_build.CSRC, src), "-o", o]))
        objs.append(o)
    assert all(p.wait() == 0 for p in procs)
    lib = str(d / "libzero_shard_hooked.so")
    arch = _build.ARCH
    subprocess.run(["nvcc", "-shared", f"-gencode=arch=compute_{arch},code=sm_{arch}", "-o", lib,
                    *objs, "-lcudart"], check=True)
    L = C.CDLL(lib)
    L.zero_test_withhold_adamw_chunk.argtypes = [C.c_ulonglong]
    L.zero_test_withhold_adamw_chunk.restype = C.c_int
    L.zero_test_squares_in_range.argtypes = [C.c_void_p, C.c_void_p, C.c_ulonglong]
    L.zero_test_squares_in_range.restype = C.c_int
    L.zero_adamw_cast_gather.argtypes = [C.POINTER(z.Layout), C.POINTER(z.HParams)] + [C.c_void_p] * 7
    L.zero_adamw_cast_gather.restype = C.c_int
    return L
