"""The sum of squares' exact-range test, on the device, against its integer definition.

The reduce pass sums squares in error-free fp32 pairs for a group of 8 values only when
every value is zero or has a magnitude in [2^-74, 2^32) (otherwise the group goes to fp64;
NaN and inf also fail, which is where the overflow flag is raised).  A wrong decision
either way is hard to see in the step's results: a group sent to fp64 without need only
costs time, and a group kept in the pair arithmetic outside its range loses exactness by
amounts far inside the norm's tolerance, or misses a NaN.  So the decision itself is
checked here: the test build's entry point runs the device test on groups built from
every exponent field, both signs, zeros, subnormals, infinities, NaNs and the values at
and next to both bounds, and each decision must equal the definition computed on the
magnitude bits as integers by numpy.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _special_values() -> np.ndarray:
    exps = np.arange(256, dtype=np.uint32) << 23
    mants = np.array([0, 1, 2, 0x3FFFFF, 0x400000, 0x7FFFFE, 0x7FFFFF], np.uint32)
    mag = (exps[:, None] | mants[None, :]).ravel()
    edges = np.array([0x1A800000, 0x4F800000], np.uint32)  # 2^-74 and 2^32
    mag = np.concatenate([mag, edges - 1, edges, edges + 1, [0, 1, 0x7F800000, 0x7FC00000]])
    return np.concatenate([mag, mag | np.uint32(0x80000000)]).astype(np.uint32)


def _expected(bits: np.ndarray) -> np.ndarray:
    u = bits & np.uint32(0x7FFFFFFF)
    ok = ((u == 0) | (u >= 0x1A800000)) & (u < 0x4F800000)
    return ok.all(axis=1)


def test_range_test_matches_its_integer_definition(hooked):
    rng = np.random.default_rng(2024)
    special = _special_values()
    n = 1 << 20
    # most groups mix special values with in-range ones, so each group's outcome turns on
    # one or two values; some are all special, some all random bit patterns
    pick = rng.choice(special, size=(n, 8))
    inrange = rng.integers(0x1A800000, 0x4F800000, size=(n, 8), dtype=np.uint32)
    inrange |= rng.integers(0, 2, size=(n, 8), dtype=np.uint32) << np.uint32(31)
    mode = rng.integers(0, 4, size=(n, 1))
    share = np.array([0.05, 1.0, 0.15, 0.125])[mode]  # the special values' share per group
    keep = rng.random((n, 8)) < share
    bits = np.where(keep, pick, inrange).astype(np.uint32)
    bits[: n // 16] = rng.integers(0, 1 << 32, size=(n // 16, 8), dtype=np.uint64).astype(np.uint32)
    bits[n // 16: n // 16 + 64] = 0  # all zero (also -0 below)
    bits[n // 16 + 64: n // 16 + 128] = 0x80000000
    want = _expected(bits)
    assert 0.2 < want.mean() < 0.8  # both outcomes well represented
    x = torch.from_numpy(bits.view(np.float32).reshape(-1)).cuda()
    out = torch.empty(n, dtype=torch.uint8, device="cuda")
    assert hooked.zero_test_squares_in_range(x.data_ptr(), out.data_ptr(), n) == 0
    got = out.cpu().numpy().astype(bool)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, [[hex(int(b)) for b in bits[i]] for i in bad[:3]]
