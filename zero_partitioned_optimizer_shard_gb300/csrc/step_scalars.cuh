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

/* Skip decision, t, decay and the loss scaler of the step being finalised (everything
 * that does not need the norm).  `overflow`: the step's reduced gradient held inf/NaN;
 * `t_next` = st->t + 1, the step count if the step is applied. */
__device__ __forceinline__ void scaler_update(zero_step_state_t* st, const zero_adamw_hparams_t& hp,
                                              uint32_t n_ranks, uint32_t overflow, uint32_t t_next)
{
    st->inv_scale_used = st->inv_scale;  // this step's unscale, for a re-reading AdamW
    float L = st->loss_scale;
    if (overflow) {
        st->skip = 1;
        st->n_skipped += 1;
        if (st->dynamic) {
            const float half = L * 0.5f;
            L = half < 1.0f ? 1.0f : half;
            st->good_steps = 0;
        }
    } else {
        st->t = t_next;
        st->skip = 0;
        st->decay = (float)(1.0 - (double)hp.lr * (double)hp.weight_decay);
        if (st->dynamic && st->growth_interval > 0) {
            st->good_steps += 1;
            if (st->good_steps == st->growth_interval) {
                const float twice = L * 2.0f;
                L = twice > 16777216.0f ? 16777216.0f : twice;
                st->good_steps = 0;
            }
        }
    }
    st->loss_scale = L;
    st->inv_scale = (float)(1.0 / ((double)n_ranks * (double)L));
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
