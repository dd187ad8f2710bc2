"""The C-ABI library without a GPU: it loads, exports every declared symbol, its host-only
layout arithmetic matches the oracle, and invalid calls are rejected on the host before
anything touches the device.

Every call below that names a device entry point is INVALID by construction, so it
returns before any CUDA call; the fake addresses in them are never dereferenced.
"""
import ctypes as C
import os
import re
import subprocess

import pytest

import oracle
import zero_partitioned_optimizer_shard_gb300 as z
from zero_partitioned_optimizer_shard_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return z.lib()


def _declared():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn), encoding="utf-8").read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(zero_\w+)\s*\(", text, flags=re.M)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 12 and "zero_step" in names and "zero_partition" in names
    out = subprocess.run(["nm", "-D", "--defined-only", z.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(lib, n)


def test_struct_sizes_match_header(lib):
    assert C.sizeof(z.StepState) == 128
    lay = z.zero_partition(1000, 4)
    assert lay.n_ranks == 4 and lay.tile_elems == z.ZERO_TILE_ELEMS


@pytest.mark.parametrize("stage", [0, 1, 2, 3])
def test_partition_matches_oracle(lib, stage):
    orc = oracle.load()
    cases = [(p, n, a) for p in (1, 2, 3, 7, 8, 63, 64, 65, 299, 1000, 1_000_003)
             for n in (1, 2, 3, 4, 5, 8, 16, 17, 64, 100) for a in (1, 8)]
    cases += [(1_557_611_200, 8, 1), (6_738_415_616, 8, 1), (2 ** 28, 16, 1), (2 ** 31 + 1, 64, 1),
              (7_500_000_000, 64, 1), (10 ** 12, 1024, 1)]
    for psi, n, a in cases:
        lz = z.zero_partition(psi, n, stage, a)
        lo = orc.partition(psi, n, stage, a)
        assert (lz.psi, lz.shard, lz.psi_padded, lz.pad) == (lo.psi, lo.shard, lo.psi_padded, lo.pad)
        assert list(lz.bytes_per_rank) == list(lo.bytes_per_rank)
        assert list(lz.comm_elems_per_rank) == list(lo.comm_elems_per_rank)
        assert lz.tiles_per_rank == -(-lz.shard // z.ZERO_TILE_ELEMS) + 1
        assert lz.n_tiles == n * lz.tiles_per_rank
        assert z.zero_workspace_bytes(lz) == 8 * lz.n_tiles


def test_partition_buckets(lib):
    lay = z.zero_partition(6_738_415_616, 8, 3, 1, 1 << 27)
    assert lay.bucket_elems == 1 << 27 and lay.n_buckets == 51
    lay = z.zero_partition(100, 4, 2, 1, 0)
    assert lay.bucket_elems == lay.psi_padded and lay.n_buckets == 1
    lay = z.zero_partition(100, 4, 2, 1, 10 ** 9)
    assert lay.bucket_elems == lay.psi_padded
    with pytest.raises(z.ZeroError):
        z.zero_partition(100, 4, 2, 1, 12)  # not a multiple of 8


@pytest.mark.parametrize("args", [(0, 4, 2, 1), (10, 0, 2, 1), (10, 4, 4, 1), (10, 4, 2, 0),
                                  (2 ** 57, 4, 2, 1), (10, 2 ** 20 + 1, 2, 1)])
def test_partition_rejects(lib, args):
    with pytest.raises(z.ZeroError) as e:
        z.zero_partition(*args)
    assert e.value.status == z.ZERO_EINVAL


# ------------------------------------------------------------------------------------------
# host-side rejection of invalid device calls (no CUDA call is reached)
# ------------------------------------------------------------------------------------------
A = 0x100000  # a 16-byte-aligned fake address; never dereferenced (every call is invalid)


def _reduce(lib, lay, dtype=z.ZERO_BF16, reps=None, begin=0, count=None, g=A, part=A, st=A):
    n = lay.n_ranks
    reps = [A] * n if reps is None else reps
    arr = (C.c_void_p * max(len(reps), 1))(*reps)
    count = lay.psi_padded if count is None else count
    return lib.zero_reduce_shard_unscale(C.byref(lay), dtype, arr, begin, count, g, part, st, None)


def test_step_launches_host_decisions(lib):
    """zero_step_launches answers on the host, without touching a GPU, for every layout
    the single launch cannot take: invalid inputs, several buckets, more than 128 tile
    slots per rank."""
    with pytest.raises(z.ZeroError) as e:
        z.zero_step_launches(z.zero_partition(1000, 4), 3)
    assert e.value.status == z.ZERO_EINVAL
    with pytest.raises(z.ZeroError):
        z.zero_step_launches(z.zero_partition(1000, 65), z.ZERO_BF16)  # > 64 ranks in kernels
    llama = z.zero_partition(6_738_415_616, 8, 3, 1, 1 << 27)
    assert z.zero_step_launches(llama, z.ZERO_BF16) == llama.n_buckets + 2 == 53
    gpt2 = z.zero_partition(1_557_611_200, 8, 2)
    assert gpt2.tiles_per_rank > 128 and z.zero_step_launches(gpt2, z.ZERO_F16) == 3


def test_reduce_rejections(lib):
    lay = z.zero_partition(1000, 4)
    assert _reduce(lib, lay, dtype=3) == z.ZERO_EINVAL
    assert _reduce(lib, lay, reps=[A, A, 0, A]) == z.ZERO_EINVAL       # a missing rank
    assert _reduce(lib, lay, count=0) == z.ZERO_EINVAL
    assert _reduce(lib, lay, begin=8, count=lay.psi_padded) == z.ZERO_EINVAL  # past the end
    assert _reduce(lib, lay, begin=lay.psi_padded, count=1) == z.ZERO_EINVAL
    assert _reduce(lib, lay, g=0) == z.ZERO_EINVAL
    assert _reduce(lib, lay, begin=4, count=8) == z.ZERO_EALIGN
    assert _reduce(lib, lay, g=A + 4) == z.ZERO_EALIGN
    assert _reduce(lib, lay, reps=[A, A + 2, A, A]) == z.ZERO_EALIGN
    assert _reduce(lib, lay, st=A + 8) == z.ZERO_EALIGN
    big = z.zero_partition(1000, 65)
    assert _reduce(lib, big) == z.ZERO_EINVAL                          # > 64 ranks in kernels
    bad = z.zero_partition(1000, 4)
    bad.psi_padded += 4                                                # corrupted layout
    assert _reduce(lib, bad) == z.ZERO_EINVAL
    bad = z.zero_partition(1000, 4)
    bad.n_tiles += 1
    assert _reduce(lib, bad) == z.ZERO_EINVAL


def test_norm_adamw_step_rejections(lib):
    lay = z.zero_partition(1000, 4)
    hp = z.hparams()
    bad_hps = [z.hparams(beta1=1.0), z.hparams(beta2=-0.1), z.hparams(eps=0.0),
               z.hparams(lr=float("nan")), z.hparams(lr=-1.0), z.hparams(weight_decay=float("inf")),
               z.hparams(params_dtype=3)]
    for b in bad_hps:
        assert lib.zero_grad_norm(C.byref(lay), C.byref(b), A, A, None) == z.ZERO_EINVAL
        assert lib.zero_adamw_cast_gather(C.byref(lay), C.byref(b), A, A, A, A, A, A, None) == z.ZERO_EINVAL
    assert lib.zero_grad_norm(C.byref(lay), C.byref(hp), 0, A, None) == z.ZERO_EINVAL
    assert lib.zero_grad_norm(C.byref(lay), C.byref(hp), A + 8, A, None) == z.ZERO_EALIGN
    assert lib.zero_adamw_cast_gather(C.byref(lay), C.byref(hp), A, A, A, 0, A, A, None) == z.ZERO_EINVAL
    assert lib.zero_adamw_cast_gather(C.byref(lay), C.byref(hp), A, A, A, A, A + 2, A, None) == z.ZERO_EALIGN
    hs = lib.zero_adamw_cast_gather_host_state
    hs.argtypes, hs.restype = lib.zero_adamw_cast_gather.argtypes, C.c_int
    for b in bad_hps:
        assert hs(C.byref(lay), C.byref(b), A, A, A, A, A, A, None) == z.ZERO_EINVAL
    assert hs(C.byref(lay), C.byref(hp), A, A, 0, A, A, A, None) == z.ZERO_EINVAL
    assert hs(C.byref(lay), C.byref(hp), A, A + 4, A, A, A, A, None) == z.ZERO_EALIGN
    # an address that is not page-locked host memory known to CUDA is refused before any
    # launch (here: no GPU, or a made-up address)
    assert hs(C.byref(lay), C.byref(hp), A, A, A, A, A, A, None) == z.ZERO_EINVAL
    reps = (C.c_void_p * 4)(A, A, A, A)
    # a bad bucket pointer anywhere rejects the whole step before any launch
    assert lib.zero_step(C.byref(lay), C.byref(hp), z.ZERO_BF16, reps, A, A, A, A, A, A + 1, A, None) == z.ZERO_EALIGN
    # g = NULL (the re-reading schedule) only for N = 2 with one window
    assert lib.zero_step(C.byref(lay), C.byref(hp), z.ZERO_BF16, reps, None, A, A, A, A, A, A, None) == z.ZERO_EINVAL
    lay2b = z.zero_partition(1 << 20, 2, 2, 1, 1 << 16)
    reps2 = (C.c_void_p * (2 * lay2b.n_buckets))(*([A] * (2 * lay2b.n_buckets)))
    assert lib.zero_step(C.byref(lay2b), C.byref(hp), z.ZERO_BF16, reps2, None, A, A, A, A, A, A, None) == z.ZERO_EINVAL
    lay2 = z.zero_partition(1000, 2)
    reps1 = (C.c_void_p * 2)(A, A)
    assert lib.zero_step(C.byref(lay2), C.byref(hp), z.ZERO_BF16, reps1, None, A, A, A, A, A + 2, A, None) == z.ZERO_EALIGN
    reps0 = (C.c_void_p * 4)(A, 0, A, A)
    assert lib.zero_step(C.byref(lay), C.byref(hp), z.ZERO_BF16, reps0, A, A, A, A, A, A, A, None) == z.ZERO_EINVAL
    assert lib.zero_step_state_init(C.byref(lay), 0.0, 1, 1000, A, A, None) == z.ZERO_EINVAL
    assert lib.zero_step_state_init(C.byref(lay), float("inf"), 1, 1000, A, A, None) == z.ZERO_EINVAL
    assert lib.zero_step_state_init(C.byref(lay), 1.0, 1, 1000, A + 4, A, None) == z.ZERO_EALIGN
    assert lib.zero_step_state_read(0, C.byref(z.StepState()), None) == z.ZERO_EINVAL


def test_step_host_rejections(lib):
    lay = z.zero_partition(1 << 20, 4, 2, 1, 1 << 16)
    hp = z.hparams()
    hreps = (C.c_void_p * 4)(A, A, A, A)
    need = 2 * 4 * (1 << 16) * 2
    args = lambda staging_bytes, s, cs: (C.byref(lay), C.byref(hp), z.ZERO_BF16, hreps, A,
                                         staging_bytes, A, A, A, A, A, A, A, None, s, cs)
    assert lib.zero_step_host(*args(need - 16, 0x10, 0x20)) == z.ZERO_ENOMEM
    assert lib.zero_step_host(*args(need, 0x10, 0x10)) == z.ZERO_EINVAL  # same stream twice
    hreps0 = (C.c_void_p * 4)(A, A, 0, A)
    assert lib.zero_step_host(C.byref(lay), C.byref(hp), z.ZERO_BF16, hreps0, A, need, A, A, A,
                              A, A, A, A, None, 0x10, 0x20) == z.ZERO_EINVAL
    # one bucket whose length is not a multiple of 8: each staged copy's slot is rounded up
    # to 8 elements (16-byte aligned copies), so staging needs 2 * N * round8(W) elements
    odd = z.zero_partition(1_000_003, 4, 2, 1, 0)
    W = odd.bucket_elems
    assert odd.n_buckets == 1 and W % 8 == 4
    no_g = lambda staging_bytes: (C.byref(odd), C.byref(hp), z.ZERO_BF16, hreps, A, staging_bytes,
                                  0, A, A, A, A, A, A, None, 0x10, 0x20)
    assert lib.zero_step_host(*no_g(2 * 4 * W * 2)) == z.ZERO_ENOMEM
    assert lib.zero_step_host(*no_g(2 * 4 * (W + 4) * 2)) == z.ZERO_EINVAL  # size passes; g = NULL


def test_strerror(lib):
    for s in (0, -1, -2, -3, -4, -5, -99):
        assert isinstance(lib.zero_strerror(s), bytes) and lib.zero_strerror(s)


def test_local_entry_point_rejections(lib):
    """The rank-local calls check the rank range, the window and the origin's alignment
    on the host."""
    lay = z.zero_partition(1000, 4, 2, 8)          # S = 256: origins 0, 256, 512, 768
    S = lay.shard
    red = lib.zero_reduce_shard_unscale_local
    red.argtypes = [C.POINTER(z.Layout), C.c_int, C.c_uint32, C.c_uint32, C.POINTER(C.c_void_p),
                    C.c_uint64, C.c_uint64, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
    red.restype = C.c_int
    reps = (C.c_void_p * 4)(A, A, A, A)
    r = lambda rb, rc, begin, count, g=A, lay=lay: red(C.byref(lay), z.ZERO_BF16, rb, rc, reps,
                                                       begin, count, g, A, A, None)
    assert r(1, 0, S, S) == z.ZERO_EINVAL          # no ranks
    assert r(4, 1, 0, S) == z.ZERO_EINVAL          # rank past N
    assert r(3, 2, 3 * S, S) == z.ZERO_EINVAL      # range past N
    assert r(1, 1, 0, S) == z.ZERO_EINVAL          # window before the range
    assert r(1, 1, S, S + 8) == z.ZERO_EINVAL      # window past the range
    assert r(1, 1, S + 4, 8) == z.ZERO_EALIGN      # window start not a multiple of 8
    assert r(1, 1, S, S, g=A + 4) == z.ZERO_EALIGN
    odd = z.zero_partition(1000, 4)                # S = 250: rank 1 starts at flat 250
    assert r(1, 1, 256, 8, lay=odd) == z.ZERO_EALIGN
    ada = lib.zero_adamw_cast_gather_local
    ada.argtypes = [C.POINTER(z.Layout), C.POINTER(z.HParams), C.c_uint32, C.c_uint32] + \
        [C.c_void_p] * 7
    ada.restype = C.c_int
    hp = z.hparams()
    assert ada(C.byref(lay), C.byref(hp), 2, 3, A, A, A, A, A, A, None) == z.ZERO_EINVAL
    assert ada(C.byref(lay), C.byref(z.hparams(eps=0.0)), 0, 1, A, A, A, A, A, A, None) == z.ZERO_EINVAL
    assert ada(C.byref(lay), C.byref(hp), 0, 1, A, A, 0, A, A, A, None) == z.ZERO_EINVAL
    assert ada(C.byref(lay), C.byref(hp), 0, 1, A, A, A, A, A + 2, A, None) == z.ZERO_EALIGN
    assert ada(C.byref(odd), C.byref(hp), 1, 1, A, A, A, A, A, A, None) == z.ZERO_EALIGN


def test_static_workspace_host_contract(lib):
    """zero_step_static_workspace has no re-reading schedule (g must be given), and g can
    stand in as zero_step_state_init's partials exactly when 4*psi_padded bytes cover the
    workspace: for every shard size S >= 4, never for S = 2 or 3."""
    f = lib.zero_step_static_workspace
    f.argtypes = [C.POINTER(z.Layout), C.POINTER(z.HParams), C.c_int, C.POINTER(C.c_void_p)] + \
        [C.c_void_p] * 7
    f.restype = C.c_int
    lay = z.zero_partition(1000, 2)
    reps = (C.c_void_p * 2)(A, A)
    hp = z.hparams()
    assert f(C.byref(lay), C.byref(hp), z.ZERO_BF16, reps, None, A, A, A, A, A, None) == z.ZERO_EINVAL
    for n in (1, 2, 4, 8, 64):
        for s_ in (1, 2, 3, 4, 5, 8, 8191, 8192, 8193, 100_000):
            L = z.zero_partition(n * s_, n)
            assert L.shard == s_
            covers = 4 * L.psi_padded >= z.zero_workspace_bytes(L)
            assert covers == (s_ >= 4), (n, s_)
