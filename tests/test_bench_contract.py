"""bench.py's command-line contract.  Without a GPU: the reference arm (the CPU oracle)
prints exactly one JSON line with the agreed keys, on one process and under torchrun with
two ranks (rank 0 prints; the other rank exits 0 without work).  On the GPU: the rank
path under torchrun (two processes sharing the one GPU over gloo) prints its line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline",
        "e2e"}


def _lines(out: str):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _check(line, n):
    assert KEYS <= set(line), KEYS - set(line)
    assert line["impl"] == "reference" and line["n_gpus"] == n and line["steps"] == 1
    assert line["value"] > 0 and line["unit"] == "params/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert "workload" in line["config"]


def test_reference_arm_one_process():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _lines(r.stdout)
    assert len(lines) == 1
    _check(lines[0], 1)


def test_reference_arm_under_torchrun_two_ranks():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
                        str(port), "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _lines(r.stdout)
    assert len(lines) == 1  # rank 0 only
    _check(lines[0], 2)


def test_reference_arm_names_each_workload():
    for wl, psi, n in (("c1", 1_000_003, 4), ("llama-7b", 6_738_415_616, 8)):
        r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                            "--warmup", "3", "--workload", wl], cwd=ROOT, capture_output=True,
                           text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        lines = _lines(r.stdout)
        assert len(lines) == 1
        _check(lines[0], 1)
        c = lines[0]["config"]
        assert c["psi"] == psi and c["n_ranks"] == n


@pytest.mark.gpu
def test_rank_path_under_torchrun_two_processes_on_one_gpu():
    """bench.py --gpus 2 runs the step with the ranks spread over two processes (here both
    on the one GPU, exchanging over gloo through host memory): one JSON line from rank 0,
    strong scaling, the per-part times and a final state after every step applied."""
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
                        str(port), "bench.py", "--gpus", "2", "--dist-backend", "gloo",
                        "--psi", str((1 << 20) + 12345), "--steps", "3", "--warmup", "3",
                        "--e2e-steps", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = _lines(r.stdout)
    assert len(lines) == 1
    line = lines[0]
    assert line["n_gpus"] == 2 and line["scaling"] == "strong" and line["value"] > 0
    assert set(line["parts_ms"]) == {"gradients", "norm inputs", "norm", "adamw", "parameters"}
    assert line["final_state"]["t"] == 3 + 3 + 3  # warm-up, timed and breakdown steps
    assert line["e2e"]["value"] > 0 and line["gpu_launches"] == 3 * 3
