"""The oracle's step on a pool of processes (the timed CPU baseline) computes what the
serial oracle step computes: the same g, master, m, v and parameters bit for bit, and the
same norm up to the grouping of the fp64 sum of squares."""
import numpy as np
import pytest

import oracle
import synth
from oracle.parallel import CHUNK, ParallelOracle
from synth import workloads as W


@pytest.mark.parametrize("wl", [W.scaled(W.C2, 3 * CHUNK + 12_345, steps=2),
                                W.scaled(W.C1, 2 * CHUNK + 7, steps=2)])
def test_parallel_oracle_equals_serial_oracle(wl):
    orc = oracle.load()
    lay = orc.partition(wl.psi, wl.n_ranks, wl.stage)
    P = lay.psi_padded
    reps = [synth.fill_host(wl.grad_out, wl.grad_kind, wl.grad_key(1, k), 0, P, wl.psi,
                            wl.grad_sigma, wl.loss_scale) for k in range(wl.n_ranks)]
    f = lambda role, kind, sig: synth.fill_host(synth.OUT_F32, kind, wl.state_key(role), 0, P,
                                                wl.psi, sig)
    master = f(synth.ROLE_MASTER, synth.NORMAL, wl.master_sigma)
    if wl.random_moments:
        m, v = f(synth.ROLE_MOM, synth.NORMAL, wl.mom_sigma), f(synth.ROLE_VAR, synth.NORMAL_SQ, wl.mom_sigma)
    else:
        m, v = np.zeros(P, np.float32), np.zeros(P, np.float32)
    g, out = np.zeros(P, np.float32), np.zeros(P, np.uint16)
    sc = oracle.scaler(wl.loss_scale, wl.dynamic, wl.growth_interval)
    hp = oracle.hparams(**wl.hp.__dict__)
    dt = oracle.F16 if wl.grad_dtype == "f16" else oracle.BF16
    with ParallelOracle(wl, procs=3) as par:
        for _ in range(2):  # the same gradients twice: the state moves on
            rep = orc.step(lay, hp, dt, reps, g, master, m, v, out, sc)
            got = par.step()
            assert got["t"] == rep.t and got["overflow"] == rep.overflow
            assert abs(got["norm"] - rep.norm) <= 1e-12 * rep.norm
            assert got["clip_coef"] == pytest.approx(rep.clip_coef, rel=2 ** -23)
            if got["clip_coef"] == rep.clip_coef:
                for name, want in (("g", g), ("master", master), ("m", m), ("v", v), ("out", out)):
                    assert np.array_equal(par.arrs[name].view(np.uint8), want.view(np.uint8)), name
