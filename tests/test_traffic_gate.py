"""bench.py reports k_adamw's DRAM traffic from committed ncu counters only while the
kernel's code is the one those counters were taken on: the gate hashes the code with its
comments and whitespace removed, so a comment edit keeps the figure and a code edit voids
it."""
import json
import os

import bench

CSRC = os.path.join(bench.ROOT, "zero_partitioned_optimizer_shard_gb300", "csrc")
FILES = [os.path.join(CSRC, n) for n in ("adamw.cu", "adamw_elem.cuh")]


def test_traffic_only_for_the_code_the_counters_were_taken_on():
    with open(os.path.join(bench.ROOT, "profiles", "k_adamw_traffic.json")) as f:
        rec = json.load(f)
    t = bench._traffic_from_profile(1_557_611_200)
    if bench.kernel_code_hash(FILES).startswith(rec["source_sha256_prefix"]):
        assert t is not None and abs(t / (30 * 1_557_611_200) - 1) < 0.01
    else:
        assert t is None  # the kernel changed since the capture: no figure


def test_hash_ignores_comments_but_not_code(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("/* one */ int f(int x) { return x + 1; } // two\n")
    h0 = bench.kernel_code_hash([str(a)])
    a.write_text("/* another\n comment */ int f(int x)  {\n return x + 1; }\n")
    assert bench.kernel_code_hash([str(a)]) == h0
    a.write_text("int f(int x) { return x + 2; }\n")
    assert bench.kernel_code_hash([str(a)]) != h0
