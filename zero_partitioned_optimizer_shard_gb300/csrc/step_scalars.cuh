/*
 * step_scalars.cuh -- the scalar part of one finalised step, shared by the norm kernel
 * (finalize.cu) and the single-launch step for small layouts (fused.cu), so both apply
 * the same policy with the same bits:
 *   - the loss scaler and skip decision of fp16 mixed-precision training ("3、ZeRO技术概述"
 *     DeepSpeed config, "fp16": enabled): a step whose reduced gradient holds inf/NaN is
 *     skipped (t unchanged) and a dynamic scale halves (floor 1); every growth_interval
 *     consecutive good steps it doubles (cap 2^24);
 *   - the bias corrections of Adam at step t, in fp64, rounded to fp32 once;
 *   - the clip coefficient of the global gradient norm (Megatron distributed-optimizer
 *     page, sec. 1): c = min(1, max_norm / (norm + 1e-6)), 1 when skipped or disabled.
 */
#pragma once

#include "zero_internal.h"

#include <math.h>

namespace zero {
namespace {

/* beta^e in fp64 by binary exponentiation: about log2(e) squarings and popcount(e)
 * multiplications, each correctly rounded.  On GB300's narrow fp64 pipe this chain is
 * about 2 us shorter than pow(), whose result it matches to a few ulp (the bias
 * corrections are rounded to fp32 once, as with pow). */
__device__ __forceinline__ double pow_uint(double beta, uint32_t e)
{
    double r = 1.0;
    while (e) {
        if (e & 1u)
            r *= beta;
        e >>= 1;
        if (e)
            beta *= beta;
    }
    return r;
}

/* lr / (1 - beta1^t) and sqrt(1 - beta2^t), each rounded to fp32 once. */
__device__ __forceinline__ float bias_step_size(const zero_adamw_hparams_t& hp, uint32_t t)
{
    return (float)((double)hp.lr / (1.0 - pow_uint((double)hp.beta1, t)));
}

__device__ __forceinline__ float bias_rbc2(const zero_adamw_hparams_t& hp, uint32_t t)
{
    return (float)sqrt(1.0 - pow_uint((double)hp.beta2, t));
}

/* The decoupled weight decay factor 1 - lr*wd, in fp64, rounded to fp32 once. */
__device__ __forceinline__ float decoupled_decay(const zero_adamw_hparams_t& hp)
{
    return (float)(1.0 - (double)hp.lr * (double)hp.weight_decay);
}

/* The scaler's outcome for either value of the step's overflow flag, computed from the
 * state before the step (it needs no norm, so it can be formed ahead of time):
 *   overflow:  the dynamic scale halves (floor 1), the good-step count restarts;
 *   no overflow: the good-step count grows and every growth_interval good steps the
 *   dynamic scale doubles (cap 2^24); the decoupled decay 1 - lr*wd;
 * and the unscale factor f32(1 / (N*L)) of the next step's reduce in each case. */
struct ScalerCand {
    float L_skip, inv_skip;
    float L_ok, inv_ok;
    uint32_t good_ok;
    float decay;
};

__device__ __forceinline__ ScalerCand scaler_candidates(const zero_step_state_t& s,
                                                        const zero_adamw_hparams_t& hp,
                                                        uint32_t n_ranks)
{
    ScalerCand c;
    const float L = s.loss_scale;
    c.L_skip = L;
    if (s.dynamic) {
        const float half = L * 0.5f;
        c.L_skip = half < 1.0f ? 1.0f : half;
    }
    c.L_ok = L;
    c.good_ok = s.good_steps;
    if (s.dynamic && s.growth_interval > 0) {
        c.good_ok = s.good_steps + 1;
        if (c.good_ok == s.growth_interval) {
            const float twice = L * 2.0f;
            c.L_ok = twice > 16777216.0f ? 16777216.0f : twice;
            c.good_ok = 0;
        }
    }
    c.inv_skip = (float)(1.0 / ((double)n_ranks * (double)c.L_skip));
    c.inv_ok = (float)(1.0 / ((double)n_ranks * (double)c.L_ok));
    c.decay = decoupled_decay(hp);
    return c;
}

/* Skip decision, t, decay and the loss scaler of the step being finalised, from its
 * candidates.  `overflow`: the step's reduced gradient held inf/NaN; `t_next` = st->t + 1,
 * the step count if the step is applied. */
__device__ __forceinline__ void scaler_apply(zero_step_state_t* st, const ScalerCand& c,
                                             uint32_t overflow, uint32_t t_next)
{
    st->inv_scale_used = st->inv_scale;  // this step's unscale, for a re-reading AdamW
    if (overflow) {
        st->skip = 1;
        st->n_skipped += 1;
        if (st->dynamic)
            st->good_steps = 0;
        st->loss_scale = c.L_skip;
        st->inv_scale = c.inv_skip;
    } else {
        st->t = t_next;
        st->skip = 0;
        st->decay = c.decay;
        st->good_steps = c.good_ok;
        st->loss_scale = c.L_ok;
        st->inv_scale = c.inv_ok;
    }
}

/* Both together: everything that does not need the norm. */
__device__ __forceinline__ void scaler_update(zero_step_state_t* st, const zero_adamw_hparams_t& hp,
                                              uint32_t n_ranks, uint32_t overflow, uint32_t t_next)
{
    const ScalerCand c = scaler_candidates(*st, hp, n_ranks);
    scaler_apply(st, c, overflow, t_next);
}

/* c = min(1, max_norm / (norm + 1e-6)) in fp64, rounded to fp32 once; 1 when the step is
 * skipped or clipping is disabled (max_norm <= 0). */
__device__ __forceinline__ float clip_coefficient(double norm, uint32_t skip, float max_norm)
{
    float c = 1.0f;
    if (!skip && max_norm > 0.0f) {
        const double cc = (double)max_norm / (norm + 1e-6);
        c = cc < 1.0 ? (float)cc : 1.0f;
    }
    return c;
}

}  // namespace
}  // namespace zero
