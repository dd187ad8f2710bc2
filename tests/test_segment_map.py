"""zero_segment_map (host-only library code) against the oracle and the hand-worked maps.

Which rank owns which piece of every model tensor: the bucketing at partition boundaries
of the ZeRO paper's gradient partitioning.  Runs without a GPU.
"""
import ctypes as C

import numpy as np
import pytest

import oracle
import zero_partitioned_optimizer_shard_gb300 as z
from synth import workloads as W
from tests import oracle_pins
from zero_partitioned_optimizer_shard_gb300 import _build


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return z.lib()


def _rows(segs):
    return [[s.tensor, s.rank, s.tensor_offset, s.shard_offset, s.count] for s in segs]


def test_hand_worked_examples(lib):
    for psi, n, sizes, want in oracle_pins._segment_cases():
        assert _rows(z.zero_segment_map(z.zero_partition(psi, n), sizes)) == want


def test_random_lists_match_oracle(lib):
    orc = oracle.load()
    rng = np.random.default_rng(5)
    for _ in range(200):
        n = int(rng.integers(1, 70))
        k = int(rng.integers(1, 40))
        sizes = [int(x) for x in rng.integers(0, 3000, k) * rng.integers(0, 2, k)]
        sizes[-1] += 1
        psi = sum(sizes)
        align = int(rng.choice([1, 8, 64]))
        got = _rows(z.zero_segment_map(z.zero_partition(psi, n, 2, align), sizes))
        want = orc.segment_map(orc.partition(psi, n, 2, align), sizes).tolist()
        assert got == want


def test_gpt2_1_5b_at_eight_ranks_matches_oracle(lib):
    """The GPT-2-1.5B buffer at N = 8: 580 tensors, 7 of them cut by a shard boundary."""
    sizes = [n for _, n in W.tensors_gpt2_1_5b()]
    orc = oracle.load()
    want = orc.segment_map(orc.partition(W.PSI_GPT2_1_5B, 8), sizes)
    got = _rows(z.zero_segment_map(z.zero_partition(W.PSI_GPT2_1_5B, 8), sizes))
    assert got == want.tolist()
    assert len(got) == len(sizes) + 7


@pytest.mark.parametrize("n", [8, 64])
def test_llama_7b_pieces_tile_every_shard(lib, n):
    """Llama-7B at N = 8 and 64: the pieces tile [0, psi) in flat order without gaps, each
    inside one shard, and each tensor's pieces tile the tensor."""
    tensors = W.tensors_llama_7b()
    sizes = [e for _, e in tensors]
    lay = z.zero_partition(W.PSI_LLAMA_7B, n)
    segs = z.zero_segment_map(lay, sizes)
    S = lay.shard
    starts = np.cumsum([0] + sizes)
    flat = 0
    per_tensor = [0] * len(sizes)
    for s in segs:
        f = s.rank * S + s.shard_offset
        assert f == flat == starts[s.tensor] + s.tensor_offset
        assert s.count >= 1 and s.shard_offset + s.count <= S
        assert s.tensor_offset == per_tensor[s.tensor]
        per_tensor[s.tensor] += s.count
        flat += s.count
    assert flat == W.PSI_LLAMA_7B and per_tensor == sizes


def test_rejections(lib):
    lay = z.zero_partition(100, 4)
    n = C.c_uint64(77)
    sizes = (C.c_uint64 * 2)(60, 40)
    f = lib.zero_segment_map
    assert f(C.byref(lay), (C.c_uint64 * 2)(60, 39), 2, None, 0, C.byref(n)) == z.ZERO_EINVAL
    assert f(C.byref(lay), (C.c_uint64 * 2)(2 ** 64 - 1, 101), 2, None, 0, C.byref(n)) == z.ZERO_EINVAL
    assert f(C.byref(lay), None, 2, None, 0, C.byref(n)) == z.ZERO_EINVAL
    assert f(C.byref(lay), sizes, 2, None, 0, None) == z.ZERO_EINVAL
    bad = z.zero_partition(100, 4)
    bad.shard += 1
    assert f(C.byref(bad), sizes, 2, None, 0, C.byref(n)) == z.ZERO_EINVAL
    # psi = 100, N = 4: S = 25; [60, 40] -> 3 pieces of tensor 0, 2 of tensor 1
    want = [[0, 0, 0, 0, 25], [0, 1, 25, 0, 25], [0, 2, 50, 0, 10], [1, 2, 0, 10, 15],
            [1, 3, 15, 0, 25]]
    assert f(C.byref(lay), sizes, 2, None, 0, C.byref(n)) == z.ZERO_OK and n.value == 5
    out = (z.Segment * 5)()
    out[4].count = 12345
    assert f(C.byref(lay), sizes, 2, out, 4, C.byref(n)) == z.ZERO_ENOMEM and n.value == 5
    assert out[0].count == 0 and out[4].count == 12345  # untouched
    assert f(C.byref(lay), sizes, 2, out, 5, C.byref(n)) == z.ZERO_OK
    assert _rows(out) == want
    with pytest.raises(z.ZeroError):
        z.zero_segment_map(lay, [10, 20])
