"""The single-launch step releases its blocks before the exact fp64 norm when an fp32
bound, rounded upwards, already shows c = min(1, max_norm / (norm + 1e-6)) = 1 (see
clip_certainly_one in the CUDA source).  That shortcut must never claim c = 1 where the
oracle's clip coefficient is below 1.  A host restatement of the bound (C, fp32 with
upward rounding, the device's constants read from the source) is checked against the
oracle on norms within 1e-9 .. 1e-3 relative of the threshold on both sides, and shown
to decide c = 1 for norms comfortably below it."""
import ctypes as C
import math
import os
import re
import subprocess

import numpy as np

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _constants():
    src = open(os.path.join(ROOT, "zero_partitioned_optimizer_shard_gb300", "csrc", "fused.cu")).read()
    m = re.search(r"need = __fmul_ru\(__fadd_ru\(__fmul_ru\(b, ([0-9.e+-]+)f\), ([0-9.e+-]+)f\), "
                  r"([0-9.e+-]+)f\)", src)
    assert m, "the bound's expression in fused.cu changed: update this test"
    return [float(np.float32(x)) for x in m.groups()]


def _model(tmp_path):
    lib = str(tmp_path / "libbound.so")
    subprocess.run(["gcc", "-O1", "-frounding-math", "-fno-fast-math", "-std=c11", "-fPIC", "-shared",
                    "-o", lib, os.path.join(ROOT, "tests", "early_release_bound.c"), "-lm"], check=True)
    L = C.CDLL(lib)
    L.certainly_one.argtypes = [C.c_float] * 5
    L.certainly_one.restype = C.c_int
    L.round_up_f32.argtypes = [C.c_double]
    L.round_up_f32.restype = C.c_float
    return L


def test_early_release_bound_never_contradicts_the_oracle(tmp_path):
    k1, k2, k3 = _constants()
    L = _model(tmp_path)
    orc = oracle.load()
    rng = np.random.default_rng(5)
    max_norms = [1e-4, 0.25, 0.5, 1.0, 3.0, 1e3] + list(rng.uniform(1e-3, 10.0, 24))
    rels = [s * 10.0 ** e for e in range(-9, -2) for s in (-1.0, -3.0, 1.0, 3.0)] + [0.0]
    certain = near = 0
    for mn in max_norms:
        mf = float(np.float32(mn))
        for rel in rels:
            norm = (mf - 1e-6) * (1.0 + rel)
            if norm <= 0.0:
                continue
            for total in (norm * norm, np.nextafter(norm * norm, math.inf), np.nextafter(norm * norm, 0.0)):
                u = L.round_up_f32(total)
                c = orc.clip_coef(math.sqrt(total), mf)
                if L.certainly_one(u, mf, k1, k2, k3):
                    certain += 1
                    assert c == 1.0, (mf, rel, total, c)
                    if abs(rel) < 1e-6:
                        near += 1
                elif rel <= -1e-5:
                    raise AssertionError(f"bound undecided far below the threshold: {mf} {rel}")
    # decided for every norm 1e-5 or more below the threshold, never within 1e-6 of it
    # unless c = 1 anyway
    assert certain > 0 and near == 0
    # and random totals far from any threshold
    for _ in range(2000):
        mf = float(np.float32(rng.uniform(1e-3, 10.0)))
        total = float(rng.uniform(0.0, 4.0 * mf * mf))
        c = orc.clip_coef(math.sqrt(total), mf)
        if L.certainly_one(L.round_up_f32(total), mf, k1, k2, k3):
            assert c == 1.0, (mf, total, c)
