"""The gradient exchange's plan across processes, checked without a GPU: how each
process's range is cut into windows, and which window each process sends and receives
at each exchange (zero_partitioned_optimizer_shard_gb300.ranks: exchange_windows,
exchange_plan, local_ranks)."""
import itertools

import pytest

import zero_partitioned_optimizer_shard_gb300 as z
from zero_partitioned_optimizer_shard_gb300 import _build
from zero_partitioned_optimizer_shard_gb300.ranks import exchange_plan, exchange_windows, local_ranks


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()  # zero_partition is host-only code in the library

CASES = [(psi, n, world, w) for psi in (13, 48_761, 100_003, 1_000_003, 3_000_017)
         for n in (2, 4, 8, 16) for world in (1, 2, 4, 8) if n % world == 0
         for w in (0, 8192, 1 << 16, 1 << 20)]


def _layout(psi, n):
    return z.zero_partition(psi, n, 2, 8)


@pytest.mark.parametrize("psi,n,world,w", CASES)
def test_windows_cover_each_range_on_the_grid(psi, n, world, w):
    lay = _layout(psi, n)
    L = lay.shard * (n // world)
    wins = exchange_windows(L, world, w)
    assert len(wins) == world
    for q, ws in enumerate(wins):
        # an exact cover of [q*L, (q+1)*L), in order, cut only at multiples of w
        assert ws[0][0] == q * L and sum(c for _, c in ws) == L
        for (b0, c0), (b1, _) in zip(ws, ws[1:]):
            assert b0 + c0 == b1 and (w == 0 or b1 % w == 0)
        assert all(c > 0 for _, c in ws)
        if w:
            assert all(c <= w for _, c in ws)


@pytest.mark.parametrize("psi,n,world,w", [c for c in CASES if c[3] != 1 << 16])
def test_no_tile_is_split_between_windows(psi, n, world, w):
    """Tiles of the sums of squares are a shard cut at the flat multiples of 8192; a
    window boundary inside a process's range is a multiple of w (itself a multiple of
    8192), so every tile lies in one window and its partial gets one add, as in the
    one-GPU step."""
    lay = _layout(psi, n)
    S, L = lay.shard, lay.shard * (n // world)
    wins = exchange_windows(L, world, w)
    for r in range(n):
        lo, hi = r * S, (r + 1) * S
        cuts = sorted(set([lo, hi] + [c for c in range((lo // 8192 + 1) * 8192, hi, 8192)]))
        for t0, t1 in zip(cuts, cuts[1:]):
            q = r // (n // world)
            inside = [(b, c) for b, c in wins[q] if b <= t0 and t1 <= b + c]
            assert len(inside) == 1, (r, t0, t1)


@pytest.mark.parametrize("psi,n,world,w", [c for c in CASES if c[2] > 1])
def test_every_send_meets_a_receive_of_its_size(psi, n, world, w):
    lay = _layout(psi, n)
    R = n // world
    L = lay.shard * R
    wins = exchange_windows(L, world, w)
    part = max(c for ws in wins for _, c in ws)
    K = max(len(ws) for ws in wins)
    received = [0] * world
    for k in range(K):
        plans = [exchange_plan(wins, p, k, R, part) for p in range(world)]
        for p, q in itertools.permutations(range(world), 2):
            sent = [(j, b, c) for (peer, j, b, c) in plans[p][0] if peer == q]
            got = [(j, o, c) for (peer, j, o, c) in plans[q][1] if peer == p]
            assert [(j, c) for j, _, c in sent] == [(j, c) for j, _, c in got]
            for (j, b, c), (_, o, _) in zip(sent, got):
                # p sends q's k-th window of its copy j; q puts it at p's place in its slot
                assert (b, c) == wins[q][k] and o == p * part and o + c <= world * part
            received[q] += sum(c for _, _, c in got)
    # every process receives (world - 1) copies of its whole range per local copy
    assert received == [(world - 1) * R * L] * world


def test_local_ranks():
    assert local_ranks(8, 2, 1) == (4, 4)
    assert local_ranks(8, 8, 7) == (7, 1)
    for bad in ((8, 3, 0), (8, 2, 2), (8, 0, 0)):
        with pytest.raises(ValueError):
            local_ranks(*bad)
