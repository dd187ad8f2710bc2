"""The boundary is a C ABI: plain C programs compiled with gcc against include/zero.h and
linked with libzero_shard.so.  tests/c_abi_host.c calls the host-only entry points (no
GPU); tests/c_abi_step.c (GPU test) runs two steps with CUDA-runtime buffers and checks
them against the C oracle on the same inputs, with no PyTorch or Python in the loop."""
import os
import subprocess

import pytest

import oracle
from zero_partitioned_optimizer_shard_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_links_and_runs(tmp_path):
    lib = _build.build()
    exe = str(tmp_path / "c_abi_host")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi_host.c"), "-o", exe,
                    "-L", os.path.dirname(lib), "-lzero_shard",
                    f"-Wl,-rpath,{os.path.dirname(lib)}"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok")
    # the Python binding's step state has the header's layout, field by field
    from zero_partitioned_optimizer_shard_gb300 import STATE_BYTES, StepState
    fields = {}
    for line in r.stdout.splitlines():
        if line.startswith("state "):
            _, name, off = line.split()
            fields[name] = int(off)
        elif line.startswith("state_size "):
            assert int(line.split()[1]) == STATE_BYTES == 128
    assert [n for n, _ in StepState._fields_] == list(fields)
    for name, off in fields.items():
        assert getattr(StepState, name).offset == off, name


def _cuda_home():
    for p in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        if p and os.path.exists(os.path.join(p, "include", "cuda_runtime.h")):
            return p
    pytest.skip("CUDA toolkit headers not found")


@pytest.mark.gpu
def test_c_program_runs_a_step_against_the_c_oracle(tmp_path):
    lib = _build.build()
    olib = oracle.build()
    cuda = _cuda_home()
    exe = str(tmp_path / "c_abi_step")
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-ffp-contract=off",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "oracle"),
                    "-I", os.path.join(cuda, "include"),
                    os.path.join(ROOT, "tests", "c_abi_step.c"), "-o", exe,
                    "-L", os.path.dirname(lib), "-lzero_shard", f"-Wl,-rpath,{os.path.dirname(lib)}",
                    olib, f"-Wl,-rpath,{os.path.dirname(olib)}",
                    "-L", os.path.join(cuda, "lib64"), "-lcudart",
                    f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}", "-lm"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok"), r.stdout



def _build_ranks_program(tmp_path):
    lib = _build.build()
    cuda = _cuda_home()
    exe = str(tmp_path / "c_abi_ranks")
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-Werror",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    os.path.join(ROOT, "tests", "c_abi_ranks.c"), "-o", exe,
                    "-L", os.path.dirname(lib), "-lzero_shard", f"-Wl,-rpath,{os.path.dirname(lib)}",
                    "-L", os.path.join(cuda, "lib64"), "-lcudart",
                    f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"], check=True)
    return exe


def test_c_program_of_the_rank_local_step_compiles(tmp_path):
    assert os.path.exists(_build_ranks_program(tmp_path))


@pytest.mark.gpu
def test_c_program_runs_the_rank_local_step_over_two_processes(tmp_path):
    """tests/c_abi_ranks.c: two processes of two ranks each through the rank-local entry
    points, exchanging by cudaMemcpy, equal to zero_step bit for bit."""
    exe = _build_ranks_program(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok"), r.stdout
