"""The synthetic workloads of the ZeRO optimizer step: shapes, seeds and distributions.

Input recipes only (what each buffer is filled with); no optimizer arithmetic.  Every
value is regenerated from (seed, role, step, rank, flat index) by the counter-based
generator in this package, on the device for the CUDA path and on the host for the
oracle, so full-size workloads never need to be copied between the two.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import synth

# GPT-2 1.5B: 48 layers, d=1600, ffn 6400, vocab 50257, 1024 positions, tied head,
# final LayerNorm.  Per layer: QKV 3d^2+3d, proj d^2+d, MLP 2*d*ffn+ffn+d, 2 LayerNorms 4d.
_D2, _FF2 = 1600, 6400
_LAYER_GPT2 = 3 * _D2 * _D2 + 3 * _D2 + _D2 * _D2 + _D2 + 2 * _D2 * _FF2 + _FF2 + _D2 + 4 * _D2
PSI_GPT2_1_5B = 48 * _LAYER_GPT2 + 50257 * _D2 + 1024 * _D2 + 2 * _D2
# Llama 7B: 32 layers, d=4096, ffn 11008, vocab 32000, untied head, RMSNorm weights.
# Per layer: q,k,v,o 4d^2, gate/up/down 3*d*ffn, 2 norms 2d.
_D7, _FF7 = 4096, 11008
_LAYER_LLAMA = 4 * _D7 * _D7 + 3 * _D7 * _FF7 + 2 * _D7
PSI_LLAMA_7B = 32 * _LAYER_LLAMA + 2 * 32000 * _D7 + _D7

assert PSI_GPT2_1_5B == 1_557_611_200
assert PSI_LLAMA_7B == 6_738_415_616



def tensors_gpt2_1_5b() -> list[tuple[str, int]]:
    """(name, elements) of GPT-2 1.5B's tensors in checkpoint order (the flat buffer's
    order): token and position embeddings, 48 blocks, the final LayerNorm; the LM head is
    tied to the token embedding."""
    d, ff = _D2, _FF2
    t = [("wte", 50257 * d), ("wpe", 1024 * d)]
    for i in range(48):
        h = f"h.{i}."
        t += [(h + "ln_1.weight", d), (h + "ln_1.bias", d),
              (h + "attn.c_attn.weight", d * 3 * d), (h + "attn.c_attn.bias", 3 * d),
              (h + "attn.c_proj.weight", d * d), (h + "attn.c_proj.bias", d),
              (h + "ln_2.weight", d), (h + "ln_2.bias", d),
              (h + "mlp.c_fc.weight", d * ff), (h + "mlp.c_fc.bias", ff),
              (h + "mlp.c_proj.weight", ff * d), (h + "mlp.c_proj.bias", d)]
    return t + [("ln_f.weight", d), ("ln_f.bias", d)]


def tensors_llama_7b() -> list[tuple[str, int]]:
    """(name, elements) of Llama 7B's tensors in checkpoint order: embedding, 32 blocks
    (attention q/k/v/o, MLP gate/up/down, two RMSNorm weights), final norm, untied head."""
    d, ff = _D7, _FF7
    t = [("embed_tokens.weight", 32000 * d)]
    for i in range(32):
        h = f"layers.{i}."
        t += [(h + f"self_attn.{x}_proj.weight", d * d) for x in "qkvo"]
        t += [(h + "mlp.gate_proj.weight", ff * d), (h + "mlp.up_proj.weight", ff * d),
              (h + "mlp.down_proj.weight", d * ff),
              (h + "input_layernorm.weight", d), (h + "post_attention_layernorm.weight", d)]
    return t + [("norm.weight", d), ("lm_head.weight", 32000 * d)]


assert sum(n for _, n in tensors_gpt2_1_5b()) == PSI_GPT2_1_5B
assert sum(n for _, n in tensors_llama_7b()) == PSI_LLAMA_7B

F16_POS_INF, F16_NAN, F16_NEG_INF = 0x7C00, 0x7E00, 0xFC00


@dataclass(frozen=True)
class HP:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    max_grad_norm: float = 1.0
    params_dtype: int = 0           # gathered parameters: 0 = bf16, 1 = fp16


@dataclass(frozen=True)
class Workload:
    name: str
    psi: int
    n_ranks: int
    stage: int
    grad_dtype: str                 # "f16" | "bf16"
    grad_kind: int                  # synth.NORMAL | synth.STUDENT_T3
    grad_sigma: float
    loss_scale: float               # initial L
    dynamic: bool                   # dynamic loss scaling (fp16)
    steps: int
    seed: int
    random_moments: bool            # m ~ N(0, 1e-4), v = N(0, 1e-4)^2; else m = v = 0
    bucket_elems: int = 0           # 0: one window over the whole flat buffer
    growth_interval: int = 1000
    master_sigma: float = 0.02
    mom_sigma: float = 1e-4
    inject_every: int = 0           # non-finite value into one replica every k-th step
    inject_rank: int = 0
    inject_base: int = 0            # at flat index base + step
    hp: HP = field(default_factory=HP)

    @property
    def grad_out(self) -> int:
        return synth.OUT_F16 if self.grad_dtype == "f16" else synth.OUT_BF16

    def grad_key(self, step: int, rank: int) -> int:
        return synth.key(self.seed, synth.ROLE_GRAD, step, rank)

    def state_key(self, role: int) -> int:
        return synth.key(self.seed, role, 0, 0)

    def injection(self, step: int):
        """(rank, flat index, fp16 bits) injected at this step, or None."""
        if not self.inject_every or step % self.inject_every:
            return None
        k = step // self.inject_every - 1
        bits = (F16_POS_INF, F16_NAN, F16_NEG_INF)[k % 3]
        return self.inject_rank, self.inject_base + step, bits


C1 = Workload("C1 odd-size fp16: psi=1,000,003, N=4, ZeRO-2", 1_000_003, 4, 2, "f16",
              synth.NORMAL, 1e-3, 1024.0, True, 1, seed=0, random_moments=False)
C2 = Workload("C2 GPT-2-1.5B flat buffer: psi=1,557,611,200, N=8, ZeRO-2, bf16 grads ~N(0,1e-4)",
              PSI_GPT2_1_5B, 8, 2, "bf16", synth.NORMAL, 1e-4, 1.0, False, 10, seed=2,
              random_moments=True)
C3 = Workload("C3 Llama-7B flat buffer: psi=6,738,415,616, N=8, ZeRO-3, 2^27-element buckets",
              PSI_LLAMA_7B, 8, 3, "bf16", synth.NORMAL, 1e-4, 1.0, False, 2, seed=3,
              random_moments=True, bucket_elems=1 << 27)
C5 = Workload("C5 fp16 dynamic-scale stress: psi=2^28, N=16, Student-t(3)*1e-3, L0=65536",
              1 << 28, 16, 2, "f16", synth.STUDENT_T3, 1e-3, 65536.0, True, 50, seed=5,
              random_moments=False, inject_every=7, inject_rank=5, inject_base=12345)


def sweep_point(psi: int, n_ranks: int, stage: int, steps: int = 1) -> Workload:
    """C4: bandwidth sweep point, bf16 grads ~N(0, 1e-3)."""
    return Workload(f"C4 sweep psi={psi} N={n_ranks} stage={stage}", psi, n_ranks, stage, "bf16",
                    synth.NORMAL, 1e-3, 1.0, False, steps, seed=4, random_moments=True)


SWEEP_PARITY_POINTS = (
    [(1 << 20, n, st) for n in (2, 4, 8, 16, 64) for st in (1, 2, 3)]
    + [((1 << 20) + 1, n, 2) for n in (2, 4, 8, 16, 64)]
    + [(1 << 24, n, 2) for n in (2, 4, 8, 16, 64)]
    + [((1 << 24) + 1, n, 2) for n in (2, 4, 8, 16, 64)])


# above 2^24 the sweep points are checked by sampling: a subset of N, elements on windows
SWEEP_SAMPLED_POINTS = [(psi, n, 2) for k in (27, 29, 31) for psi in (1 << k, (1 << k) + 1)
                        for n in (2, 8, 64)]


def sweep_name(psi: int, n_ranks: int, stage: int) -> str:
    return f"C4-{psi}-{n_ranks}-{stage}"


def by_name(name: str) -> Workload:
    """C1, C2, C3, C5, or a sweep point "C4-<psi>-<N>-<stage>" (two steps; 2^27-element
    buckets when the N gradient copies would not fit beside the state in ~200 GB)."""
    if name.startswith("C4-"):
        _, psi, n, st = name.split("-")
        from dataclasses import replace
        wl = sweep_point(int(psi), int(n), int(st), steps=2)
        P = -(-wl.psi // wl.n_ranks) * wl.n_ranks
        if wl.n_ranks * P * 2 + 18 * P > 200e9:
            wl = replace(wl, bucket_elems=1 << 27)
        return wl
    return globals()[name]


def scaled(w: Workload, psi: int, steps: int | None = None, name: str | None = None) -> Workload:
    """The same recipe at another size (small parity cases of a large workload)."""
    from dataclasses import replace
    return replace(w, psi=psi, steps=w.steps if steps is None else steps,
                   name=name or f"{w.name.split(':')[0]} scaled to psi={psi}")
