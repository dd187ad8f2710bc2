"""The boundary is a C ABI: a plain C program (tests/c_abi_host.c) compiled with gcc against
include/zero.h and linked with libzero_shard.so calls the host-only entry points.  No GPU
is touched."""
import os
import subprocess

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
