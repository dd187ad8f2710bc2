"""The seeded input generator (host twin): casts, distributions, determinism.  No GPU."""
import numpy as np
import pytest

import synth
from synth import workloads as W


def _edge_f32():
    rng = np.random.default_rng(0)
    u = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    # values around every binary16 rounding regime: subnormals, the normal range, overflow
    mags = np.concatenate([rng.uniform(-30, 17, 100000)])
    v = (np.sign(rng.uniform(-1, 1, mags.size)) * 2.0 ** mags).astype(np.float32)
    # exact binary16 ties: odd multiples of half a binary16 ulp
    h16 = rng.integers(0, 0x7BFF, 20000).astype(np.uint16).view(np.float16)
    up16 = np.nextafter(h16, np.float16(np.inf))
    ties = ((h16.astype(np.float64) + up16.astype(np.float64)) / 2).astype(np.float32)
    edge = np.array([65504, 65519.99, 65520, 65536, 2 ** -24, 2 ** -25, 2 ** -25 * 1.0000001,
                     3 * 2 ** -26, 2 ** -14, 2 ** -14 * (1 - 2 ** -11), 0.0, -0.0, np.inf, -np.inf],
                    np.float32)
    x = np.concatenate([u.view(np.float32), v, ties, edge, -edge])
    return x[~np.isnan(x)]


def test_f16_cast_matches_numpy():
    x = _edge_f32()
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)  # numpy: IEEE round-to-nearest-even
    got = np.array([synth.host().zsynth_f32_to_f16(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref), np.flatnonzero(got != ref)[:10]


def test_bf16_cast_matches_torch():
    import torch
    x = _edge_f32()
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([synth.host().zsynth_f32_to_bf16(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)


def test_normal_moments():
    n = 1 << 21
    z = synth.fill_host(synth.OUT_F32, synth.NORMAL, synth.key(9, 1, 1, 0), 0, n, n, 1.0)
    assert abs(z.mean()) < 5 / np.sqrt(n)
    assert abs(z.var() - 1.0) < 5 * np.sqrt(2.0 / n)
    assert np.abs(z).max() <= 6.0
    # Irwin-Hall(12) has excess kurtosis -0.1
    k = np.mean(z.astype(np.float64) ** 4) / np.mean(z.astype(np.float64) ** 2) ** 2 - 3
    assert abs(k + 0.1) < 0.02
    # values are multiples of 2^-16 (exact integer sum scaled by a power of two)
    assert np.all(np.float64(z) * 65536 == np.round(np.float64(z) * 65536))


def test_student_t3_shape():
    n = 1 << 20
    t = synth.fill_host(synth.OUT_F32, synth.STUDENT_T3, synth.key(9, 1, 2, 0), 0, n, n, 1.0)
    # t(3): median |t| = 0.7649, P(|t| > 3.182) = 0.05
    assert abs(np.median(np.abs(t)) - 0.7649) < 0.005
    assert abs(np.mean(np.abs(t) > 3.182) - 0.05) < 0.002


def test_scale_sigma_square_and_padding():
    k = synth.key(1, 2, 0, 0)
    z = synth.fill_host(synth.OUT_F32, synth.NORMAL, k, 100, 50, 130, 1.0)
    s = synth.fill_host(synth.OUT_F32, synth.NORMAL, k, 100, 50, 130, 0.02)
    q = synth.fill_host(synth.OUT_F32, synth.NORMAL_SQ, k, 100, 50, 130, 1e-4)
    assert np.array_equal(s[:30], (z[:30] * np.float32(0.02)).astype(np.float32))
    w = (z[:30] * np.float32(1e-4)).astype(np.float32)
    assert np.array_equal(q[:30], (w * w).astype(np.float32))
    assert np.all(s[30:] == 0) and np.all(q[30:] == 0)


def test_windows_gather_and_threads_agree():
    k = synth.key(3, 1, 4, 2)
    full = synth.fill_host(synth.OUT_BF16, synth.NORMAL, k, 0, 100000, 99990, 1e-4)
    for a, b in [(0, 7), (13, 5000), (99980, 20)]:
        part = synth.fill_host(synth.OUT_BF16, synth.NORMAL, k, a, b, 99990, 1e-4)
        assert np.array_equal(part, full[a:a + b])
    idx = np.array([0, 5, 99989, 99990, 31337], np.uint64)
    assert np.array_equal(synth.gather_host(synth.OUT_BF16, synth.NORMAL, k, idx, 99990, 1e-4),
                          full[idx.astype(np.int64)])


def test_workload_sizes():
    assert W.C2.psi == 1_557_611_200 and W.C3.psi == 6_738_415_616 and W.C5.psi == 2 ** 28
    assert [W.C5.injection(s) for s in (6, 7, 14, 21, 28)] == [
        None, (5, 12352, 0x7C00), (5, 12359, 0x7E00), (5, 12366, 0xFC00), (5, 12373, 0x7C00)]


@pytest.mark.parametrize("sigma,scale", [(1e-3, 1024.0), (1e-4, 1.0)])
def test_fp16_grads_reasonable(sigma, scale):
    x = synth.fill_host(synth.OUT_F16, synth.NORMAL, synth.key(0, 1, 1, 0), 0, 1 << 16, 1 << 16,
                        sigma, scale).view(np.float16).astype(np.float64)
    assert abs(x.std() - sigma * scale) < 0.02 * sigma * scale
