"""Planted mistakes in the oracle must be caught by its pins.

Each case copies the oracle's C source, changes one line the way a plausible slip would
(a dropped term, a wrong sign or index, a transposed operand, an off-by-one), builds it
into a temporary library and runs every pin against it.  At least one pin must fail.
The mistakes live only in temporary copies on the CPU.
"""
import os

import pytest

import oracle
from tests import oracle_pins

MUTANTS = [
    # number formats
    ("f16 subnormal scale", "mag = ldexpf((float)f, -24);", "mag = ldexpf((float)f, -25);"),
    ("f16 exponent bias", "mag = ldexpf((float)(1024 + f), e - 25);",
     "mag = ldexpf((float)(1024 + f), e - 24);"),
    ("bf16 ties away from zero", "if (low > 0x8000u || (low == 0x8000u && (kept & 1u)))",
     "if (low >= 0x8000u)"),
    ("bf16 decode shift", "uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    ("f16 ties away", "float r = nearbyintf(q);", "float r = roundf(q);"),
    ("f16 unit", "float unit = ldexpf(1.0f, exp16 - 10);", "float unit = ldexpf(1.0f, exp16 - 9);"),
    ("f16 subnormal threshold", "if (a == 0.0f || exp16 < -14)", "if (a == 0.0f || exp16 < -15)"),
    # partition / ledger / communication
    ("shard floor", "uint64_t S = (psi + n_ranks - 1) / n_ranks;", "uint64_t S = psi / n_ranks + 1;"),
    ("align ignored", "S = (S + align - 1) / align * align;", "S = S;"),
    ("stage-1 ledger", "out->bytes_per_rank[1] = 2 * P + 2 * P + 12 * S;",
     "out->bytes_per_rank[1] = 2 * P + 2 * S + 12 * S;"),
    ("stage-2 ledger", "out->bytes_per_rank[2] = 2 * P + 2 * S + 12 * S;",
     "out->bytes_per_rank[2] = 2 * P + 2 * P + 12 * S;"),
    ("stage-3 ledger", "out->bytes_per_rank[3] = 2 * S + 2 * S + 12 * S;",
     "out->bytes_per_rank[3] = 2 * S + 2 * S + 12 * P;"),
    ("ring rounds", "uint64_t ring = (n_ranks - 1) * S;", "uint64_t ring = n_ranks * S;"),
    ("stage-3 traffic", "out->comm_elems_per_rank[3] = 3 * ring;",
     "out->comm_elems_per_rank[3] = 2 * ring;"),
    # reduce-scatter
    ("owner index", "uint64_t owner = i / lay->shard;", "uint64_t owner = i % lay->n_ranks;"),
    ("descending rank sum", "for (uint64_t k = 0; k < lay->n_ranks; ++k)\n                s = s + replica_value",
     "for (uint64_t k = lay->n_ranks; k-- > 0;)\n                s = s + replica_value"),
    ("dropped rank", "for (uint64_t k = 0; k < lay->n_ranks; ++k)\n                s = s + replica_value",
     "for (uint64_t k = 1; k < lay->n_ranks; ++k)\n                s = s + replica_value"),
    ("no unscale", "gi = s * inv_scale;", "gi = s;"),
    ("pad read", "if (i < lay->psi) {", "if (i <= lay->psi) {"),
    ("sumsq not squared", "sumsq[owner] += (double)gi * (double)gi;", "sumsq[owner] += (double)gi;"),
    ("flag inverted", "if (!isfinite(gi))\n            *overflow = 1;", "if (isnan(gi))\n            *overflow = 1;"),
    ("inv without N", "return (float)(1.0 / ((double)n_ranks * (double)loss_scale));",
     "return (float)(1.0 / (double)loss_scale);"),
    # norm / clip
    ("norm not rooted", "return sqrt(q);\n}\n\n/* [MD] sec. 1: the global norm determines",
     "return q;\n}\n\n/* [MD] sec. 1: the global norm determines"),
    ("norm drops last rank", "for (uint64_t r = 0; r < n_ranks; ++r)\n        q = q + sumsq[r];",
     "for (uint64_t r = 0; r + 1 < n_ranks; ++r)\n        q = q + sumsq[r];"),
    ("clip eps sign", "double c = (double)max_norm / (norm + 1e-6);",
     "double c = (double)max_norm / (norm - 1e-6);"),
    ("clip comparison", "return c < 1.0 ? (float)c : 1.0f;", "return c > 1.0 ? (float)c : 1.0f;"),
    # per-tensor segment map
    ("segment rank", "uint64_t r = i / lay->shard;", "uint64_t r = i / (lay->shard + 1);"),
    ("segment shard offset", "out[n].shard_offset = i - r * lay->shard;",
     "out[n].shard_offset = i - start_of_k;"),
    ("segment tensor offset", "out[n].tensor_offset = i - start_of_k;", "out[n].tensor_offset = i;"),
    ("segment ignores shard cuts", "if (k != cur_tensor || r != cur_rank) {", "if (k != cur_tensor) {"),
    ("segment size check", "if (total != lay->psi)", "if (total > lay->psi)"),
    # scaler
    ("backoff factor", "float half = s->loss_scale * 0.5f;", "float half = s->loss_scale * 0.25f;"),
    ("t on overflow", "        s->n_skipped += 1;\n        return 0;", "        s->n_skipped += 1;\n        s->t += 1;\n        return 0;"),
    ("growth off by one", "if (s->good_steps == s->growth_interval) {",
     "if (s->good_steps > s->growth_interval) {"),
    ("no growth reset", "            s->good_steps = 0;\n        }\n    }\n    return 1;",
     "        }\n    }\n    return 1;"),
    # AdamW
    ("bias correction t+1", "double bc1 = 1.0 - pow((double)hp->beta1, (double)t);",
     "double bc1 = 1.0 - pow((double)hp->beta1, (double)(t + 1));"),
    ("bc2 unrooted", "*rbc2 = (float)sqrt(bc2);", "*rbc2 = (float)bc2;"),
    ("decay without lr", "*decay = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);",
     "*decay = (float)(1.0 - (double)hp->weight_decay);"),
    ("m transposed", "float m_new = b1 * *m + omb1 * gc;", "float m_new = omb1 * *m + b1 * gc;"),
    ("v not squared", "float v_new = b2 * *v + omb2 * (gc * gc);", "float v_new = b2 * *v + omb2 * gc;"),
    ("clip not applied", "float gc = c * g;", "float gc = g;"),
    ("eps inside sqrt", "float denom = sqrtf(v_new) / rbc2 + hp->eps;",
     "float denom = sqrtf(v_new / rbc2 + hp->eps);"),
    ("rbc2 multiplied", "float denom = sqrtf(v_new) / rbc2 + hp->eps;",
     "float denom = sqrtf(v_new) * rbc2 + hp->eps;"),
    ("update sign", "float p_new = *p * decay - step_size * (m_new / denom);",
     "float p_new = *p * decay + step_size * (m_new / denom);"),
    ("decay dropped", "float p_new = *p * decay - step_size * (m_new / denom);",
     "float p_new = *p - step_size * (m_new / denom);"),
    ("old moment in update", "float p_new = *p * decay - step_size * (m_new / denom);",
     "float p_new = *p * decay - step_size * (*m / denom);"),
    ("pad rule", "if (i >= lay->psi) {\n            out[i] = 0;", "if (i > lay->psi) {\n            out[i] = 0;"),
    ("shard offset", "uint64_t lo = rank * lay->shard;\n    uint64_t hi = lo + lay->shard;",
     "uint64_t lo = rank * lay->shard;\n    uint64_t hi = lo + lay->shard - 1;"),
    # whole step
    ("replica offset", "shard_ptrs[k] = replicas[k] + r * S;", "shard_ptrs[k] = replicas[0] + r * S;"),
    ("update when skipped", "    if (applied)\n        for (uint64_t r = 0; r < N; ++r)",
     "    if (1)\n        for (uint64_t r = 0; r < N; ++r)"),
    ("stale t", "oracle_adamw_shard(lay, hp, c, sc->t, r, g, master, m, v, out);",
     "oracle_adamw_shard(lay, hp, c, sc->t + 1, r, g, master, m, v, out);"),
]


@pytest.fixture(scope="module")
def source():
    with open(oracle.SRC, encoding="utf-8") as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, source, name, old, new):
    assert source.count(old) == 1, f"mutation anchor for '{name}' not unique"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new), encoding="utf-8")
    hdr = os.path.join(os.path.dirname(oracle.SRC), "zero_oracle.h")
    (tmp_path / "zero_oracle.h").write_text(open(hdr, encoding="utf-8").read(), encoding="utf-8")
    lib = oracle.build(str(src), str(tmp_path / "libmutant.so"), force=True)
    orc = oracle.load(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, ZeroDivisionError, OverflowError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake '{name}'"
