"""Pins of the CPU oracle: checks against what the ZeRO pages and mathematics fix.

Each ``pin_*`` function takes a loaded oracle (``oracle.load(path)``) and raises
AssertionError when the oracle disagrees with a printed value, a closed form, an
invariant, a library routine or brute force.  ``test_oracle_pins.py`` runs them on the
oracle; ``test_oracle_mutants.py`` runs them on copies of the oracle with one planted
mistake each and requires that at least one pin fails for every mistake.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
U = 2.0 ** -24  # fp32 unit roundoff
F16, BF16 = 1, 2


def f32(x) -> float:
    return float(np.float32(x))


def _hp(orc_mod, **kw):
    import oracle
    return oracle.hparams(**kw)


# ------------------------------------------------------------------------------------------
# number formats
# ------------------------------------------------------------------------------------------
def pin_f16_decode_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float32)  # numpy: IEEE binary16 decode
    got = np.array([orc.f16_to_f32(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def pin_bf16_decode_all_patterns(orc):
    import torch
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = np.array([orc.bf16_to_f32(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def pin_bf16_encode_vs_torch(orc):
    import torch
    rng = np.random.default_rng(1)
    u = rng.integers(0, 2 ** 32, size=40000, dtype=np.uint64).astype(np.uint32)
    # exact ties (low half = 0x8000) with even and odd kept parts, and near-max values
    ties = (rng.integers(0, 2 ** 16, size=4000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    edge = np.array([0x7f7fffff, 0x7f7f8000, 0x7f7f7fff, 0xff7fffff, 0x00008000, 0x00018000,
                     0x7f800000, 0xff800000, 0, 0x80000000, 0x3f808000, 0x3f818000],
                    dtype=np.uint32)
    allu = np.concatenate([u, ties, edge])
    x = allu.view(np.float32)
    keep = ~np.isnan(x)
    x = x[keep]
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.f32_to_bf16(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref), int(np.sum(got != ref))
    # NaN stays NaN (quiet, sign kept)
    for b in (0x7fc00000, 0xffc00001, 0x7f800001):
        r = orc.f32_to_bf16(float(np.uint32(b).view(np.float32)))
        assert (r & 0x7f80) == 0x7f80 and (r & 0x7f) != 0 and (r >> 15) == (b >> 31)


def pin_f16_encode_vs_numpy(orc):
    rng = np.random.default_rng(2)
    u = rng.integers(0, 2 ** 32, size=30000, dtype=np.uint64).astype(np.uint32)
    mags = (np.sign(rng.uniform(-1, 1, 30000)) * 2.0 ** rng.uniform(-30, 17, 30000)).astype(np.float32)
    h16 = rng.integers(0, 0x7BFF, 6000).astype(np.uint16).view(np.float16)
    ties = ((h16.astype(np.float64) + np.nextafter(h16, np.float16(np.inf)).astype(np.float64)) / 2)
    edge = np.array([65504, 65519.99, 65520, 65536, 2 ** -24, 2 ** -25, 3 * 2 ** -26, 2 ** -14,
                     2 ** -14 * (1 - 2 ** -11), 0.0, -0.0, np.inf, -np.inf, 1.0, -2.5], np.float32)
    x = np.concatenate([u.view(np.float32), mags, ties.astype(np.float32), edge, -edge])
    x = x[~np.isnan(x)]
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)  # numpy: IEEE round-to-nearest-even
    got = np.array([orc.f32_to_f16(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref), np.flatnonzero(got != ref)[:5]
    r = orc.f32_to_f16(float("nan"))
    assert (r & 0x7c00) == 0x7c00 and (r & 0x3ff) != 0


# ------------------------------------------------------------------------------------------
# partition, ledger, communication
# ------------------------------------------------------------------------------------------
def pin_partition_bruteforce(orc):
    for align in (1, 8):
        for n in range(1, 18):
            for psi in list(range(1, 70)) + [97, 128, 255, 256, 299, 300]:
                lay = orc.partition(psi, n, 2, align)
                S, P = lay.shard, lay.psi_padded
                # brute force: the smallest multiple of align whose N copies cover psi
                s = align
                while s * n < psi:
                    s += align
                assert S == s and P == n * s and lay.pad == P - psi, (psi, n, align)
                # every flat index has exactly one owner, at offset r*S, shards contiguous
                owners = np.full(P, -1)
                for r in range(n):
                    seg = owners[r * S:(r + 1) * S]
                    assert np.all(seg == -1)
                    seg[:] = r
                assert np.all(owners >= 0)
                assert lay.n_buckets == 1 and lay.bucket_elems == P


def pin_partition_ledger_formulas(orc):
    """[ZM] sec. 3: 16, 4 + 12/N, 2 + 14/N and 16/N bytes per parameter (N | Psi)."""
    for psi, n in [(8, 4), (1024, 8), (3 * 64, 64), (10 ** 9, 8), (6, 1), (4096 * 7, 7)]:
        for stage in range(4):
            lay = orc.partition(psi, n, stage)
            b = [Fraction(int(x)) for x in lay.bytes_per_rank]
            assert b[0] == 16 * psi
            assert b[1] == (4 + Fraction(12, n)) * psi
            assert b[2] == (2 + Fraction(14, n)) * psi
            assert b[3] == Fraction(16, n) * psi
    # with padding, counted bytes never go below the formula and exceed it by at most
    # the padded elements' share
    for psi, n in [(1_000_003, 4), (17, 5), (299, 16)]:
        lay = orc.partition(psi, n, 1)
        pad = lay.pad
        b = [int(x) for x in lay.bytes_per_rank]
        assert b[0] == 16 * psi
        for got, per_param, per_shard in ((b[1], 4, 12), (b[2], 2, 14), (b[3], 0, 16)):
            exact = per_param * psi + Fraction(per_shard * psi, n)
            assert exact <= got <= exact + per_param * pad + per_shard * (pad / n + 1)


def _golden_ledger():
    rows = []
    with open(os.path.join(GOLDEN, "ledger_printed.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.split("|")[0].strip()
            if not line or line.startswith("#"):
                continue
            psi, n, stage, q, printed, check = line.split()
            rows.append((int(psi), int(n), int(stage), q, float(printed), check))
    return rows


def _matches(computed, printed, check):
    if check.startswith("d"):
        return round(computed, int(check[1:])) == printed
    return abs(computed - printed) <= float(check[1:]) * abs(computed)


def pin_ledger_printed_numbers(orc):
    for psi, n, stage, q, printed, check in _golden_ledger():
        if q == "bytes":
            gb = orc.partition(psi, n, stage).bytes_per_rank[stage] / 1e9
        else:  # largest Psi whose stage bytes fit 32 GB, by bisection on the layout
            lo, hi = 1, 10 ** 13
            while lo < hi:
                mid = (lo + hi + 1) // 2
                if orc.partition(mid, n, stage).bytes_per_rank[stage] <= 32e9:
                    lo = mid
                else:
                    hi = mid - 1
            gb = lo / 1e9
        assert _matches(gb, printed, check), (psi, n, stage, q, gb, printed)


def pin_comm_volume(orc):
    """[ZW] sec. 6(1) eq. dp-comm: a ring reduce-scatter sends (N-1)/N * Psi per rank and
    the all-gather the same: 2 Psi for DP and stages 1-2; stage 3 adds one more Psi."""
    for psi, n in [(8, 4), (7_500_000_000, 64), (1024, 2), (5, 1)]:
        lay = orc.partition(psi, n, 3)
        c = [int(x) for x in lay.comm_elems_per_rank]
        one = Fraction((n - 1) * psi, n)
        assert c[0] == c[1] == c[2] == 2 * one
        assert c[3] == 3 * one
        if n > 1:
            assert Fraction(c[3], c[2]) == Fraction(3, 2)


def pin_worked_example_8x4(orc):
    """[ZW] sec. 6(2): 8 parameters, 4 GPUs; GPU r keeps G_2r, G_2r+1 after the
    reduce-scatter, updates p_2r, p_2r+1, and the all-gather yields [p0' .. p7']."""
    import oracle
    kv = {}
    with open(os.path.join(GOLDEN, "worked_example_8x4.txt"), encoding="utf-8") as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, *vals = line.split()
                kv[k] = [int(v) for v in vals]
    psi, n, owner = kv["psi"][0], kv["n_ranks"][0], kv["owner"]
    lay = orc.partition(psi, n, 2)
    assert [i // lay.shard for i in range(psi)] == owner and lay.pad == 0
    # gradients g_kj = small integers (exact in fp16); the average is exact
    g_int = np.array([[(3 * k + 5 * j) % 11 - 5 for j in range(psi)] for k in range(n)])
    reps = [g_int[k].astype(np.float16).view(np.uint16) for k in range(n)]
    for r in range(n):
        g = np.zeros(psi, np.float32)
        sumsq = np.zeros(n, np.float64)
        ov = np.zeros(1, np.uint32)
        lo = r * lay.shard
        orc.reduce_window(lay, F16, [x[lo:] for x in reps], lo, lay.shard,
                          orc.inv_scale(n, 1.0), g[lo:], sumsq, ov)
        for j in range(psi):
            if owner[j] == r:
                assert Fraction(float(g[j])) == Fraction(int(g_int[:, j].sum()), n)
                assert sumsq[r] > 0 or np.all(g_int[:, lo:lo + lay.shard].sum(0) == 0)
            else:
                assert g[j] == 0.0 and sumsq[owner[j]] == 0.0  # nothing outside shard r
    # sharded step == unsharded step on the averaged gradient, output in [p0' .. p7'] order
    hp = oracle.hparams(max_grad_norm=0.0)
    rng = np.random.default_rng(3)
    p0 = rng.normal(0, 0.02, psi).astype(np.float32)
    a = [p0.copy(), np.zeros(psi, np.float32), np.zeros(psi, np.float32)]
    b = [p0.copy(), np.zeros(psi, np.float32), np.zeros(psi, np.float32)]
    g = np.zeros(psi, np.float32)
    out_a = np.zeros(psi, np.uint16)
    out_b = np.zeros(psi, np.uint16)
    orc.step(lay, hp, F16, reps, g, *a, out_a, oracle.scaler(1.0))
    gm = (g_int.sum(0) / n).astype(np.float32)
    orc.step_unsharded(hp, gm, *b, out_b, oracle.scaler(1.0))
    assert np.array_equal(g, gm)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    assert np.array_equal(out_a, out_b)


# ------------------------------------------------------------------------------------------
# reduce-scatter arithmetic
# ------------------------------------------------------------------------------------------
def _reduce_all(orc, lay, dtype, reps, inv):
    P, n = lay.psi_padded, lay.n_ranks
    g = np.full(P, np.nan, np.float32)
    sumsq = np.zeros(n, np.float64)
    ov = np.zeros(1, np.uint32)
    orc.reduce_window(lay, dtype, reps, 0, P, inv, g, sumsq, ov)
    return g, sumsq, int(ov[0])


def pin_reduce_integer_exact(orc):
    rng = np.random.default_rng(5)
    for n, L in [(4, 1024.0), (8, 1.0), (16, 65536.0), (3, 4.0), (5, 2.0), (7, 1.0)]:
        psi = 257
        lay = orc.partition(psi, n, 2)
        vals = rng.integers(-2048, 2049, size=(n, lay.psi_padded))
        vals[:, psi:] = 0
        for dtype, npt in ((F16, np.float16), (BF16, None)):
            if dtype == BF16:
                vals_b = rng.integers(-256, 257, size=(n, lay.psi_padded))
                vals_b[:, psi:] = 0
                reps = [_bf16_bits(vals_b[k].astype(np.float32)) for k in range(n)]
                ints = vals_b
            else:
                reps = [vals[k].astype(np.float16).view(np.uint16) for k in range(n)]
                ints = vals
            inv = orc.inv_scale(n, L)
            assert inv == f32(1.0 / (n * L))
            g, _, ov = _reduce_all(orc, lay, dtype, reps, inv)
            assert ov == 0
            s = ints.sum(0)  # exact integer sums, exact in fp32 (|s| < 2^24)
            # the reduced gradient is the exact sum times f32(1/(N*L)), rounded once
            expect = (s.astype(np.float32) * np.float32(inv)).astype(np.float32)
            assert np.array_equal(g.view(np.uint32), expect.view(np.uint32))
            if (n * L) == 2 ** round(math.log2(n * L)):
                for j in range(0, psi, 31):
                    assert Fraction(float(g[j])) == Fraction(int(s[j])) / Fraction(n) / Fraction(L)


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """Exact bf16 bit patterns of fp32 values already representable in bf16."""
    u = x.astype(np.float32).view(np.uint32)
    assert np.all((u & 0xFFFF) == 0)
    return (u >> 16).astype(np.uint16)


def pin_reduce_order_ascending(orc):
    """Ascending rank order: 1 + 2^-24 rounds back to 1 (tie to even) twice, while the
    descending order would first make 2^-23 and keep it.  Chosen reading, pinned."""
    lay = orc.partition(8, 3, 2, align=1)
    vals = np.zeros((3, lay.psi_padded), np.float32)
    vals[0, :8] = 1.0
    vals[1, :8] = 2.0 ** -24
    vals[2, :8] = 2.0 ** -24
    reps = [_bf16_bits(vals[k]) for k in range(3)]
    g, _, _ = _reduce_all(orc, lay, BF16, reps, 1.0)
    assert np.all(g[:8] == 1.0)
    vals = vals[::-1].copy()
    reps = [_bf16_bits(vals[k]) for k in range(3)]
    g, _, _ = _reduce_all(orc, lay, BF16, reps, 1.0)
    assert np.all(g[:8] == np.float32(1.0 + 2.0 ** -23))


def pin_reduce_sumsq_and_attribution(orc):
    rng = np.random.default_rng(7)
    for psi, n in [(1003, 4), (4096, 8), (77, 16), (10, 3)]:
        lay = orc.partition(psi, n, 2)
        S = lay.shard
        # rank-dependent magnitudes make a misattributed element visible
        x = np.zeros((n, lay.psi_padded), np.float32)
        for k in range(n):
            x[k, :psi] = rng.normal(0, 1, psi) * (1 + np.arange(psi) // S)
        reps = [x[k].astype(np.float16).view(np.uint16) for k in range(n)]
        inv = orc.inv_scale(n, 2.0)
        g, sumsq, ov = _reduce_all(orc, lay, F16, reps, inv)
        assert ov == 0
        for r in range(n):
            ref = math.fsum(float(v) ** 2 for v in g[r * S:(r + 1) * S].astype(np.float64))
            assert abs(sumsq[r] - ref) <= 1e-13 * max(ref, 1e-300)
        norm, tot = orc.global_norm(sumsq)
        ref_tot = math.fsum(float(v) ** 2 for v in g.astype(np.float64))
        assert abs(tot - ref_tot) <= 1e-13 * ref_tot
        assert abs(norm - math.sqrt(ref_tot)) <= 1e-13 * math.sqrt(ref_tot)


def pin_reduce_overflow_flags(orc):
    n, psi = 6, 60
    lay = orc.partition(psi, n, 2)
    base = np.ones((n, lay.psi_padded), np.float16)
    base[:, psi:] = 0
    for bad in (np.inf, -np.inf, np.nan):
        for rank, idx in ((5, 0), (0, psi - 1), (2, 17)):
            x = base.copy()
            x[rank, idx] = bad
            g, sumsq, ov = _reduce_all(orc, lay, F16, [x[k].view(np.uint16) for k in range(n)], 1.0)
            assert ov == 1 and not np.isfinite(g[idx])
            assert np.all(np.isfinite(np.delete(g, idx)))
    g, _, ov = _reduce_all(orc, lay, F16, [base[k].view(np.uint16) for k in range(n)], 1.0)
    assert ov == 0
    # bf16 inputs: an fp32 sum that overflows is caught even though every input is finite
    big = np.zeros((2, 8), np.float32)
    big[:, 3] = 3.0e38
    lay2 = orc.partition(8, 2, 2)
    g, _, ov = _reduce_all(orc, lay2, BF16, [_bf16_bits(_round_bf16(big[k])) for k in range(2)], 0.5)
    assert ov == 1 and np.isinf(g[3])


def _round_bf16(x):
    import torch
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).float().numpy()


def pin_reduce_pads_ignored(orc):
    """Padding positions carry a zero gradient whatever the replicas hold there."""
    for psi, n in [(10, 4), (5, 8), (1, 3)]:
        lay = orc.partition(psi, n, 2)
        assert lay.pad > 0
        x = np.ones((n, lay.psi_padded), np.float16)
        x[:, psi:] = np.nan
        g, sumsq, ov = _reduce_all(orc, lay, F16, [x[k].view(np.uint16) for k in range(n)], 1.0)
        assert ov == 0 and np.all(g[psi:] == 0) and np.all(g[:psi] == np.float32(n))
        assert abs(sumsq.sum() - psi * n * n) < 1e-9


def pin_reduce_windows_union(orc):
    """Bucketed windows in any split reproduce the one-window result bit for bit."""
    rng = np.random.default_rng(11)
    psi, n = 999, 4
    lay = orc.partition(psi, n, 2)
    P = lay.psi_padded
    x = rng.normal(0, 1, (n, P)).astype(np.float16)
    reps = [x[k].view(np.uint16) for k in range(n)]
    g1, s1, _ = _reduce_all(orc, lay, F16, reps, 0.25)
    cuts = sorted(set([0, P] + list(rng.integers(1, P, 7))))
    g2 = np.zeros(P, np.float32)
    s2 = np.zeros(n, np.float64)
    ov = np.zeros(1, np.uint32)
    for a, b in zip(cuts[:-1], cuts[1:]):
        orc.reduce_window(lay, F16, [r[a:] for r in reps], a, b - a, 0.25, g2[a:], s2, ov)
    assert np.array_equal(g1.view(np.uint32), g2.view(np.uint32)) and np.array_equal(s1, s2)


def pin_inv_scale(orc):
    for n, L in [(1, 1.0), (3, 1.0), (4, 1024.0), (16, 65536.0), (7, 3.0), (64, 0.5)]:
        assert orc.inv_scale(n, L) == f32(1.0 / (n * L))


# ------------------------------------------------------------------------------------------
# norm and clip
# ------------------------------------------------------------------------------------------
def pin_norm_constant_closed_form(orc):
    """Constant a in every replica: g = a/L, norm = |a|/L * sqrt(psi) (pads excluded)."""
    for psi, n, a, L in [(1000, 4, 3.0, 1024.0), (4097, 8, -0.5, 1.0), (33, 5, 2.0, 4.0)]:
        lay = orc.partition(psi, n, 2)
        x = np.zeros((n, lay.psi_padded), np.float16)
        x[:, :psi] = a
        g, sumsq, _ = _reduce_all(orc, lay, F16, [x[k].view(np.uint16) for k in range(n)],
                                  orc.inv_scale(n, L))
        gi = float(g[0])
        assert np.all(g[:psi] == np.float32(gi))
        assert abs(gi - a / L) <= 2 * U * abs(a / L)
        norm, _ = orc.global_norm(sumsq)
        assert abs(norm - abs(gi) * math.sqrt(psi)) <= 1e-12 * norm


def pin_clip_cases(orc):
    for norm, clip in [(0.5, 1.0), (0.0, 1.0), (1.0 - 2e-6, 1.0), (3.0, 1.0), (7.25, 1.0),
                       (1e6, 2.5), (2.0, 0.0), (2.0, -1.0), (10.0, 0.001)]:
        c = orc.clip_coef(norm, clip)
        if clip <= 0:
            assert c == 1.0
        else:
            ref = min(1.0, f32(clip) / (norm + 1e-6))
            assert c == f32(ref), (norm, clip, c, ref)


# ------------------------------------------------------------------------------------------
# AdamW
# ------------------------------------------------------------------------------------------
def pin_adamw_scalars(orc):
    import oracle
    hp = oracle.hparams(lr=1e-3, beta1=0.9, beta2=0.999, weight_decay=0.01)
    b1, b2, lr, wd = f32(0.9), f32(0.999), f32(1e-3), f32(0.01)
    for t in (1, 2, 7, 50, 1000):
        s, r, d = orc.adamw_scalars(hp, t)
        assert s == f32(lr / (1 - b1 ** t)) and r == f32(math.sqrt(1 - b2 ** t))
        assert d == f32(1 - lr * wd)


def pin_adamw_t1_closed_form(orc):
    """t = 1 from zero moments: m_hat = gc, v_hat = gc^2, so
    p' = p (1 - lr wd) - lr gc / (|gc| + eps), m = (1-b1) gc, v = (1-b2) gc^2."""
    import oracle
    rng = np.random.default_rng(13)
    n = 4000
    for c in (1.0, 0.37):
        hp = oracle.hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
        g = rng.normal(0, 1e-3, n).astype(np.float32)
        g[:5] = [0.0, 1e-8, -1e-8, 3e-9, 1.0]
        p = rng.normal(0, 0.02, n).astype(np.float32)
        m = np.zeros(n, np.float32)
        v = np.zeros(n, np.float32)
        out = np.zeros(n, np.uint16)
        p_in = p.copy()
        orc.adamw_elements(hp, c, 1, g, p, m, v, out)
        lr, wd, b1, b2, eps = f32(1e-3), f32(0.01), f32(0.9), f32(0.999), f32(1e-8)
        gc = f32(c) * g.astype(np.float64)
        em = (1 - b1) * gc
        ev = (1 - b2) * gc * gc
        ep = p_in.astype(np.float64) * (1 - lr * wd) - lr * gc / (np.abs(gc) + eps)
        assert np.all(np.abs(m - em) <= 3 * U * np.abs(em))
        assert np.all(np.abs(v - ev) <= 5 * U * np.abs(ev))
        assert np.all(np.abs(p - ep) <= 16 * U * (np.abs(p_in) + lr))


def pin_adamw_constant_gradient_multistep(orc):
    """Constant gradient from zero moments: bias correction makes m_hat = g and
    v_hat = g^2 at every t, so each step moves p by exactly lr*g/(|g|+eps) after the
    decoupled decay: p_T = p_0 d^T - u * sum_{k<T} d^k."""
    import oracle
    T = 40
    for wd in (0.0, 0.1):
        hp = oracle.hparams(lr=1e-2, beta1=0.9, beta2=0.99, eps=1e-8, weight_decay=wd)
        g = np.array([1e-3, -2e-2, 5.0, 3e-8, -1e-7], np.float32)
        p = np.array([0.5, -0.25, 1.0, 0.125, 0.0], np.float32)
        p0 = p.astype(np.float64)
        m = np.zeros_like(p)
        v = np.zeros_like(p)
        out = np.zeros(p.size, np.uint16)
        for t in range(1, T + 1):
            orc.adamw_elements(hp, 1.0, t, g, p, m, v, out)
        lr, eps = f32(1e-2), f32(1e-8)
        d = 1 - lr * f32(wd)
        gd = g.astype(np.float64)
        u = lr * gd / (np.abs(gd) + eps)
        expect = p0 * d ** T - u * sum(d ** k for k in range(T))
        assert np.all(np.abs(p - expect) <= 1e-5 * (np.abs(p0) + T * lr)), (p, expect)


def pin_adamw_special_cases(orc):
    import oracle
    rng = np.random.default_rng(17)
    n = 512
    g = rng.normal(0, 1e-2, n).astype(np.float32)
    p = rng.normal(0, 1, n).astype(np.float32)
    m0 = rng.normal(0, 1e-3, n).astype(np.float32)
    v0 = (rng.normal(0, 1e-3, n) ** 2).astype(np.float32)
    out = np.zeros(n, np.uint16)
    # g = 0 from zero moments: pure decoupled decay
    hp = oracle.hparams(lr=0.05, weight_decay=0.2)
    q = p.copy()
    orc.adamw_elements(hp, 1.0, 3, np.zeros(n, np.float32), q, np.zeros(n, np.float32),
                       np.zeros(n, np.float32), out)
    assert np.array_equal(q, (p * np.float32(f32(1 - f32(0.05) * f32(0.2)))).astype(np.float32))
    # lr = 0: parameters unchanged, moments still move
    hp = oracle.hparams(lr=0.0, weight_decay=0.3)
    q, m, v = p.copy(), m0.copy(), v0.copy()
    orc.adamw_elements(hp, 1.0, 5, g, q, m, v, out)
    assert np.array_equal(q, p) and not np.array_equal(m, m0) and not np.array_equal(v, v0)
    # beta1 = beta2 = 0: m = gc, v = gc^2, no bias correction
    hp = oracle.hparams(lr=1e-3, beta1=0.0, beta2=0.0, eps=1e-6, weight_decay=0.0)
    q, m, v = p.copy(), m0.copy(), v0.copy()
    orc.adamw_elements(hp, 0.5, 9, g, q, m, v, out)
    gc = 0.5 * g.astype(np.float64)
    assert np.all(np.abs(m - gc) <= U * np.abs(gc)) and np.all(np.abs(v - gc * gc) <= 3 * U * gc * gc)
    ep = p - f32(1e-3) * gc / (np.abs(gc) + f32(1e-6))
    assert np.all(np.abs(q - ep) <= 8 * U * (np.abs(p) + 1e-3))
    # general step from random moments vs the fp64 formula (tolerance from rounding)
    hp = oracle.hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    q, m, v = p.copy(), m0.copy(), v0.copy()
    t, c = 4, 0.8
    orc.adamw_elements(hp, c, t, g, q, m, v, out)
    b1, b2, lr, eps, wd = f32(0.9), f32(0.999), f32(1e-3), f32(1e-8), f32(0.01)
    gc = f32(c) * g.astype(np.float64)
    em = b1 * m0 + (1 - b1) * gc
    ev = b2 * v0 + (1 - b2) * gc * gc
    ep = p * (1 - lr * wd) - lr / (1 - b1 ** t) * em / (np.sqrt(ev / (1 - b2 ** t)) + eps)
    scale_m = b1 * np.abs(m0) + (1 - b1) * np.abs(gc)
    assert np.all(np.abs(m - em) <= 3 * U * scale_m)
    assert np.all(np.abs(v - ev) <= 3 * U * ev)
    assert np.all(np.abs(q - ep) <= 1e-5 * (np.abs(p) + lr))


def pin_adamw_bf16_output(orc):
    import oracle
    import torch
    rng = np.random.default_rng(19)
    n = 3000
    hp = oracle.hparams()
    p = rng.normal(0, 0.02, n).astype(np.float32)
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    out = np.zeros(n, np.uint16)
    orc.adamw_elements(hp, 1.0, 1, g, p, np.zeros(n, np.float32), np.zeros(n, np.float32), out)
    ref = torch.from_numpy(p.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out, ref)


def pin_adamw_f16_output(orc):
    """The fp16 gathered-parameter variant writes numpy's binary16 of the fp32 master."""
    import oracle
    rng = np.random.default_rng(21)
    n = 3000
    hp = oracle.hparams(params_dtype=F16)
    p = rng.normal(0, 0.02, n).astype(np.float32)
    g = rng.normal(0, 1e-3, n).astype(np.float32)
    out = np.zeros(n, np.uint16)
    orc.adamw_elements(hp, 1.0, 1, g, p, np.zeros(n, np.float32), np.zeros(n, np.float32), out)
    assert np.array_equal(out, p.astype(np.float16).view(np.uint16))


def pin_adamw_shard_pads(orc):
    import oracle
    psi, n = 13, 4
    lay = orc.partition(psi, n, 2)
    P = lay.psi_padded
    hp = oracle.hparams()
    rng = np.random.default_rng(23)
    g = rng.normal(0, 1e-3, P).astype(np.float32)
    arrs = [rng.normal(0, 1, P).astype(np.float32) for _ in range(3)]
    arrs[2] = np.abs(arrs[2])
    keep = [a.copy() for a in arrs]
    out = np.full(P, 0xABCD, np.uint16)
    for r in range(n):
        orc.adamw_shard(lay, hp, 1.0, 1, r, g, *arrs, out)
    assert np.all(out[psi:] == 0)
    for a, k in zip(arrs, keep):
        assert np.array_equal(a[psi:], k[psi:])
    # real positions equal the element-wise update at the same offsets
    q = [k[:psi].copy() for k in keep]
    o2 = np.zeros(psi, np.uint16)
    orc.adamw_elements(hp, 1.0, 1, g[:psi].copy(), *q, o2)
    assert np.array_equal(out[:psi], o2)
    for a, b in zip(arrs, q):
        assert np.array_equal(a[:psi], b)


# ------------------------------------------------------------------------------------------
# scaler
# ------------------------------------------------------------------------------------------
def pin_scaler_sequences(orc):
    import oracle
    sc = oracle.scaler(65536.0, dynamic=True, growth_interval=3)
    pattern = [1, 1, 0, 0, 0, 0, 1, 0, 0, 0, 0, 0, 0]
    Ls, ts = [], []
    for ov in pattern:
        orc.scaler_update(sc, ov)
        Ls.append(sc.loss_scale)
        ts.append(sc.t)
    assert Ls == [32768, 16384, 16384, 16384, 32768, 32768, 16384, 16384, 16384, 32768,
                  32768, 32768, 65536]
    assert ts == [0, 0, 1, 2, 3, 4, 4, 5, 6, 7, 8, 9, 10] and sc.n_skipped == 3
    # floor at 1 and cap at 2^24
    sc = oracle.scaler(4.0, dynamic=True, growth_interval=1)
    for _ in range(5):
        orc.scaler_update(sc, 1)
    assert sc.loss_scale == 1.0
    sc = oracle.scaler(2.0 ** 23, dynamic=True, growth_interval=1)
    for _ in range(3):
        orc.scaler_update(sc, 0)
    assert sc.loss_scale == 2.0 ** 24
    # a static scale never changes; overflow still skips
    sc = oracle.scaler(1.0, dynamic=False)
    assert orc.scaler_update(sc, 1) == 0 and sc.loss_scale == 1.0 and sc.t == 0
    assert orc.scaler_update(sc, 0) == 1 and sc.t == 1


# ------------------------------------------------------------------------------------------
# whole steps
# ------------------------------------------------------------------------------------------
def _random_problem(psi, n, dtype, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    P = n * (-(-psi // n))
    x = np.zeros((n, P), np.float32)
    x[:, :psi] = rng.normal(0, 1e-3, (n, psi)) * scale
    if dtype == F16:
        reps = [x[k].astype(np.float16).view(np.uint16) for k in range(n)]
    else:
        reps = [_bf16_bits(_round_bf16(x[k])) for k in range(n)]
    st = [np.zeros(P, np.float32) for _ in range(3)]
    st[0][:psi] = rng.normal(0, 0.02, psi)
    st[1][:psi] = rng.normal(0, 1e-4, psi)
    st[2][:psi] = rng.normal(0, 1e-4, psi) ** 2
    return reps, st


def pin_step_identity_unsharded(orc):
    """The concatenation of the N shard updates equals the unsharded AdamW step on the
    all-reduced mean gradient ([ZS]: ZeRO-1 only splits the all-reduce in two)."""
    import oracle
    for psi, n, dtype, clip in [(1001, 4, F16, 0.0), (1001, 4, F16, 1e-3), (512, 8, BF16, 1.0),
                                (37, 16, BF16, 0.05)]:
        lay = orc.partition(psi, n, 2)
        P = lay.psi_padded
        reps, st = _random_problem(psi, n, dtype, psi + n)
        hp = oracle.hparams(max_grad_norm=clip)
        a = [s.copy() for s in st]
        g = np.zeros(P, np.float32)
        out = np.zeros(P, np.uint16)
        L = 1024.0 if dtype == F16 else 1.0
        for t in range(1, 4):
            sc_a = oracle.scaler(L, dynamic=(dtype == F16), t=t - 1)
            rep_a = orc.step(lay, hp, dtype, reps, g, *a, out, sc_a)
            b = [s[:psi].copy() for s in st] if t == 1 else b
            ob = np.zeros(psi, np.uint16)
            sc_b = oracle.scaler(L, dynamic=(dtype == F16), t=t - 1)
            rep_b = orc.step_unsharded(hp, g[:psi].copy(), *b, ob, sc_b)
            assert rep_a.overflow == rep_b.overflow == 0 and rep_a.t == rep_b.t == t
            assert abs(rep_a.norm - rep_b.norm) <= 1e-13 * rep_b.norm
            if rep_a.clip_coef == rep_b.clip_coef:
                for x, y in zip(a, b):
                    assert np.array_equal(x[:psi].view(np.uint32), y.view(np.uint32))
                assert np.array_equal(out[:psi], ob)
            else:  # fp64 sums in another order moved c by one fp32 ulp
                assert abs(rep_a.clip_coef - rep_b.clip_coef) <= 2 * U * rep_b.clip_coef
            assert np.all(out[psi:] == 0)
            # g is the mean of the replicas, unscaled
            if t == 1:
                xs = np.stack([orc_f(dtype, r) for r in reps]).astype(np.float64)
                gm = xs.sum(0)[:psi] / (n * L)
                assert np.all(np.abs(g[:psi] - gm) <= 2 * U * np.abs(gm) + 1e-30)


def orc_f(dtype, bits):
    if dtype == F16:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def pin_step_stage_independent(orc):
    import oracle
    psi, n = 333, 4
    reps, st = _random_problem(psi, n, F16, 29)
    outs = []
    for stage in (1, 2, 3):
        lay = orc.partition(psi, n, stage)
        a = [s.copy() for s in st]
        g = np.zeros(lay.psi_padded, np.float32)
        out = np.zeros(lay.psi_padded, np.uint16)
        orc.step(lay, oracle.hparams(), F16, reps, g, *a, out, oracle.scaler(1024.0, True))
        outs.append((g, a, out))
    for g, a, out in outs[1:]:
        assert np.array_equal(g, outs[0][0]) and np.array_equal(out, outs[0][2])
        for x, y in zip(a, outs[0][1]):
            assert np.array_equal(x, y)


def pin_step_skip_untouched(orc):
    import oracle
    psi, n = 200, 4
    lay = orc.partition(psi, n, 2)
    reps, st = _random_problem(psi, n, F16, 31)
    reps[2] = reps[2].copy()
    reps[2][57] = 0x7C00  # +inf in rank 2's copy
    a = [s.copy() for s in st]
    g = np.zeros(lay.psi_padded, np.float32)
    out = np.full(lay.psi_padded, 0x1234, np.uint16)
    sc = oracle.scaler(65536.0, dynamic=True, t=5)
    rep = orc.step(lay, oracle.hparams(), F16, reps, g, *a, out, sc)
    assert rep.overflow == 1 and rep.skipped == 1 and rep.t == 5 and sc.t == 5
    assert rep.loss_scale_used == 65536.0 and sc.loss_scale == 32768.0
    assert np.all(out == 0x1234)
    for x, y in zip(a, st):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


# ------------------------------------------------------------------------------------------
# per-tensor segment map
# ------------------------------------------------------------------------------------------
def _segment_cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "segment_map_examples.txt"), encoding="utf-8") as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            if line.startswith("case"):
                psi, n, *sizes = (int(x) for x in line.split()[1:])
                cur = (psi, n, sizes, [])
                cases.append(cur)
            else:
                cur[3].append([int(x) for x in line.split()])
    return cases


def pin_segment_map_examples(orc):
    """Hand-worked maps, including the 8-parameter, 4-GPU example of [ZW] sec. 6(2)."""
    for psi, n, sizes, want in _segment_cases():
        got = orc.segment_map(orc.partition(psi, n), sizes)
        assert got.tolist() == want, (psi, n, sizes, got.tolist())


def _segments_by_runs(psi, shard, sizes):
    """The same map derived another way: label every element with (tensor, rank) using
    numpy and cut where the label changes."""
    tensor = np.repeat(np.arange(len(sizes)), sizes)
    flat = np.arange(psi)
    rank = flat // shard
    start = np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64)
    cut = np.flatnonzero(np.r_[True, (tensor[1:] != tensor[:-1]) | (rank[1:] != rank[:-1])])
    ends = np.r_[cut[1:], psi]
    return [[int(tensor[c]), int(rank[c]), int(c - start[tensor[c]]), int(c - rank[c] * shard),
             int(e - c)] for c, e in zip(cut, ends)]


def pin_segment_map_runs_and_count(orc):
    rng = np.random.default_rng(11)
    for _ in range(60):
        n = int(rng.integers(1, 18))
        k = int(rng.integers(1, 30))
        sizes = [int(x) for x in rng.integers(0, 400, k)]
        sizes[int(rng.integers(0, k))] += 1  # psi >= 1
        psi = sum(sizes)
        lay = orc.partition(psi, n, 2, int(rng.choice([1, 8])))
        got = orc.segment_map(lay, sizes).tolist()
        assert got == _segments_by_runs(psi, lay.shard, sizes)
        # one piece per non-empty tensor plus one per shard boundary strictly inside a tensor
        starts = np.cumsum([0] + sizes)
        inside = sum(1 for b in range(1, n) for t in range(k)
                     if starts[t] < b * lay.shard < starts[t + 1])
        assert len(got) == sum(1 for x in sizes if x) + inside
        assert sum(row[4] for row in got) == psi


def pin_segment_map_rejects_bad_sums(orc):
    lay = orc.partition(100, 4)
    for sizes in ([99], [50, 51], [], [100, 1]):
        try:
            orc.segment_map(lay, sizes)
        except ValueError:
            continue
        raise AssertionError(f"sizes {sizes} accepted for psi=100")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
