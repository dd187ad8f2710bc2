/*
 * zero_oracle.c -- CPU oracle for the ZeRO-DP partitioned mixed-precision AdamW step.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load this library.  It shares no code
 * with the CUDA library.  Build: gcc -O2 -ffp-contract=off -fPIC -shared (no fast-math),
 * so every floating-point operation below is exactly the one written, in the order written.
 *
 * Source pages (see zero_oracle.h for the full names):
 *   [ZW] "【论文解读】ZeRO"   [ZM] "ZeRO 显存优化：ZeRO-1、ZeRO-2 与 ZeRO-3"
 *   [ZS] operatorworld.com ZeRO optimizer-sharding article
 *   [ZO] "3、ZeRO技术概述：ZeRO三个阶段原理与对比"
 *   [MD] gitcode.csdn.net article on Megatron's distributed optimizer and ZeRO
 *
 * Precision.  The pages fix the optimizer side at fp32: the master weights, momentum and
 * variance are fp32 ([ZW] sec. 2(1), [ZS] 16-byte ledger), and the reduced gradient is an
 * fp32 average of the ranks' fp16/bf16 gradients.  So the per-element reduce and AdamW
 * arithmetic is fp32, in the order written here.  Everything the pages leave free is fp64:
 * the sum of squares behind the global norm, the norm, the clip coefficient and the bias
 * corrections (rounded to fp32 once, where the fp32 element update consumes them).
 *
 * Pins (tests/test_oracle_*.py; a planted mistake in any function fails at least one):
 *   number formats        all 65536 fp16 patterns vs numpy.float16; bf16 vs torch.bfloat16
 *   oracle_partition      brute-force exact cover; the ledger numbers the pages print;
 *                         the four per-stage ledger formulas and 2/2/3-Psi traffic
 *   oracle_reduce_window  integer-valued replicas vs exact rational means; the 8-parameter,
 *                         4-GPU worked example of [ZW] sec. 6(2); math.fsum for sumsq;
 *                         injected inf/NaN; per-rank attribution with asymmetric data
 *   oracle_global_norm,
 *   oracle_clip_coef      closed forms (constant gradients), math.fsum, clip cases
 *   oracle_adamw_*        closed forms: t=1 from zero moments, constant gradient over many
 *                         steps (bias correction makes the step exactly lr*g/(|g|+eps)),
 *                         g=0 (pure decay), lr=0, beta1=beta2=0
 *   oracle_scaler_update  back-off / growth sequences in closed form
 *   oracle_step           identity: the sharded step equals the unsharded step on the
 *                         averaged gradient ([ZS]: ZeRO-1 only splits the all-reduce);
 *                         independent of the stage; skip leaves every byte untouched
 *   oracle_segment_map    hand-worked maps (one is the [ZW] sec. 6(2) example with one
 *                         tensor per parameter); a numpy run-length derivation; the count
 *                         (non-empty tensors + boundaries strictly inside a tensor)
 * Parity unpinned: none beyond the readings listed with each function (the AdamW form,
 * the clip epsilon and the scaler policy are chosen readings; their closed forms pin the
 * code to the chosen reading, not the reading to the pages).
 */
#include "zero_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------ */
/* Number formats (IEEE 754 binary16; bfloat16 = the top half of an IEEE binary32).      */
/* ------------------------------------------------------------------------------------ */

float oracle_f16_to_f32(uint16_t h)
{
    /* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits */
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    float mag;
    if (e == 0)
        mag = ldexpf((float)f, -24);              /* zero / subnormal: f * 2^-24 */
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexpf((float)(1024 + f), e - 25);  /* (1 + f/1024) * 2^(e-15) */
    return sign ? -mag : mag;
}

float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return x;
}

uint16_t oracle_f32_to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if (isnan(x))
        return (uint16_t)(((u >> 16) & 0x8000u) | 0x7fc0u);
    /* Round to nearest, ties to even, on the 16 discarded bits: the low half is compared
     * with one half-unit (0x8000); above it rounds up, below it truncates, at exactly one
     * half it rounds up only when the kept part is odd.  A carry out of the fraction moves
     * the exponent up by one, which is the correct rounding (and gives inf past the max). */
    uint32_t kept = u >> 16;
    uint32_t low = u & 0xffffu;
    if (low > 0x8000u || (low == 0x8000u && (kept & 1u)))
        kept += 1;
    return (uint16_t)kept;
}

/* IEEE binary16 from binary32, round to nearest, ties to even.  Magnitudes from 65520
 * (halfway between the largest finite binary16, 65504, and 2^16) up round to inf; below
 * 2^-14 the result is a multiple of 2^-24 (subnormal); NaN stays a quiet NaN. */
uint16_t oracle_f32_to_f16(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if (isnan(x))
        return (uint16_t)(sign | 0x7e00u);
    float a = fabsf(x);
    if (a >= 65520.0f)
        return (uint16_t)(sign | 0x7c00u);
    /* scale so that one unit in the last binary16 place becomes 1, round the scaled value
     * to an integer with ties to even, and rebuild the bits from exponent and fraction */
    int e;
    frexpf(a, &e);                 /* a = f * 2^e, f in [0.5, 1) (a > 0) */
    int exp16 = e - 1;             /* a in [2^exp16, 2^(exp16+1)) */
    if (a == 0.0f || exp16 < -14)
        exp16 = -14;               /* subnormal range: the unit is 2^-24 */
    float unit = ldexpf(1.0f, exp16 - 10);
    float q = a / unit;            /* exact: a power-of-two scaling */
    float r = nearbyintf(q);       /* round-half-even in the default rounding mode */
    uint32_t mant = (uint32_t)r;   /* up to 2048 when rounding carries into the next binade */
    if (mant == 0)
        return sign;
    if (exp16 == -14 && mant < 1024)
        return (uint16_t)(sign | mant);                      /* subnormal */
    if (mant == 2048) {
        mant = 1024;
        exp16 += 1;
    }
    return (uint16_t)(sign | (uint32_t)(exp16 + 15) << 10 | (mant - 1024));
}

static float replica_value(int dtype, uint16_t bits)
{
    return dtype == ORACLE_F16 ? oracle_f16_to_f32(bits) : oracle_bf16_to_f32(bits);
}

/* ------------------------------------------------------------------------------------ */
/* Partition, ledger and communication volume.                                          */
/* ------------------------------------------------------------------------------------ */

/* [ZW] sec. 4(1)-(3): the model states are split into N_d equal partitions and rank i
 * owns partition i.  Equal partitions of a flat buffer need padding when N does not
 * divide Psi: S = ceil(Psi/N), rounded up to `align`, and the buffer grows to N*S.
 *
 * Ledger ([ZW] sec. 2(1), [ZM] sec. 2-3, [ZS], [MD] sec. 2 table): per parameter 2 bytes
 * of fp16/bf16 weight, 2 bytes of gradient and K = 12 bytes of fp32 master, momentum and
 * variance.  Plain DP holds all of it: 16*Psi.  Stage 1 splits the optimizer states:
 * 2*Psi + 2*Psi + 12*Psi/N.  Stage 2 also splits gradients: 2*Psi + 14*Psi/N.  Stage 3
 * splits everything: 16*Psi/N.  Reading for padding: count what is allocated, i.e. full
 * buffers are N*S long and a shard is S long; with N | Psi and align = 1 this is exactly
 * the pages' formulas.
 *
 * Communication ([ZW] sec. 6(1) eq. dp-comm and 6(2)-(3), [ZS] communication accounting):
 * a ring reduce-scatter or all-gather runs N-1 rounds and each rank sends one Psi/N
 * chunk per round.  Plain DP (all-reduce = reduce-scatter + all-gather), stage 1 and
 * stage 2 send 2(N-1)S elements per rank; stage 3 adds a second parameter all-gather for
 * backward: 3(N-1)S.  For large N these are 2*Psi and 3*Psi (the 1.5x of stage 3). */
int oracle_partition(uint64_t psi, uint64_t n_ranks, uint32_t stage, uint64_t align,
                     uint64_t bucket_elems, oracle_layout_t* out)
{
    if (!out || psi == 0 || n_ranks == 0 || align == 0 || stage > 3)
        return -1;
    if (psi > (1ull << 56) || n_ranks > (1ull << 20) || align > (1ull << 20))
        return -1;
    uint64_t S = (psi + n_ranks - 1) / n_ranks;
    S = (S + align - 1) / align * align;
    uint64_t P = n_ranks * S;
    memset(out, 0, sizeof *out);
    out->psi = psi;
    out->n_ranks = n_ranks;
    out->shard = S;
    out->psi_padded = P;
    out->pad = P - psi;
    out->align = align;
    out->bucket_elems = bucket_elems ? bucket_elems : P;
    out->n_buckets = (P + out->bucket_elems - 1) / out->bucket_elems;
    out->stage = stage;
    out->bytes_per_rank[0] = 16 * psi;                /* 2 + 2 + 12 bytes per parameter */
    out->bytes_per_rank[1] = 2 * P + 2 * P + 12 * S;  /* weights, grads full; K*S */
    out->bytes_per_rank[2] = 2 * P + 2 * S + 12 * S;  /* weights full; grads and K*S */
    out->bytes_per_rank[3] = 2 * S + 2 * S + 12 * S;  /* everything sharded */
    uint64_t ring = (n_ranks - 1) * S;                /* one ring reduce-scatter or all-gather */
    out->comm_elems_per_rank[0] = 2 * ring;
    out->comm_elems_per_rank[1] = 2 * ring;
    out->comm_elems_per_rank[2] = 2 * ring;
    out->comm_elems_per_rank[3] = 3 * ring;
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Reduce-scatter arithmetic, unscale, overflow check.                                  */
/* ------------------------------------------------------------------------------------ */

float oracle_inv_scale(uint64_t n_ranks, float loss_scale)
{
    return (float)(1.0 / ((double)n_ranks * (double)loss_scale));
}

/* [ZW] sec. 6(1)-(2): data-parallel training averages the ranks' gradients; with
 * gradient partitioning the average is reduce-scattered, so rank r ends up holding only
 * the averaged gradient of its own partition [r*S, (r+1)*S) ([ZW] sec. 6(2) example:
 * GPU0 keeps G0,G1, GPU1 keeps G2,G3, ...; [ZO] "method flow", step 3; [MD] sec. 2,
 * ZeRO-2 snapshot).  Readings: the average is an fp32 sum over ranks in ascending rank
 * order; the loss scale L of fp16 training ([ZO] config "fp16": enabled) is removed in
 * the same single multiply by f32(1/(N*L)); the overflow check looks at the reduced
 * fp32 gradient; the norm's sum of squares is fp64 per rank, ascending flat index.
 * replicas[k] and g both point at flat element `begin`.
 * Padding positions (>= psi) hold a zero gradient and are not read from the replicas. */
void oracle_reduce_window(const oracle_layout_t* lay, int dtype, const uint16_t* const* replicas,
                          uint64_t begin, uint64_t count, float inv_scale, float* g,
                          double* sumsq, uint32_t* overflow)
{
    for (uint64_t i = begin; i < begin + count; ++i) {
        uint64_t owner = i / lay->shard;
        float gi = 0.0f;
        if (i < lay->psi) {
            float s = 0.0f;
            for (uint64_t k = 0; k < lay->n_ranks; ++k)
                s = s + replica_value(dtype, replicas[k][i - begin]);
            gi = s * inv_scale;
        }
        g[i - begin] = gi;
        if (!isfinite(gi))
            *overflow = 1;
        sumsq[owner] += (double)gi * (double)gi;
    }
}

/* ------------------------------------------------------------------------------------ */
/* Global gradient norm and clip coefficient.                                           */
/* ------------------------------------------------------------------------------------ */

/* [MD] sec. 1, the AdamW global grad-norm table: inside optimizer.step(), before
 * clipping, one all-reduce sums the ranks' local squared norms into the global L2 norm
 * that sets the clip coefficient.  The all-reduce here is the rank-ordered fp64 sum. */
double oracle_global_norm(const double* sumsq, uint64_t n_ranks, double* total)
{
    double q = 0.0;
    for (uint64_t r = 0; r < n_ranks; ++r)
        q = q + sumsq[r];
    if (total)
        *total = q;
    return sqrt(q);
}

/* [MD] sec. 1: the global norm determines clip_coeff.  Reading (the formula is not on
 * the pages): the usual global-norm clipping, c = min(1, max_norm / (norm + 1e-6)),
 * evaluated in fp64 and rounded to fp32 once; max_norm <= 0 disables clipping. */
float oracle_clip_coef(double norm, float max_norm)
{
    if (!(max_norm > 0.0f))
        return 1.0f;
    double c = (double)max_norm / (norm + 1e-6);
    return c < 1.0 ? (float)c : 1.0f;
}

/* ------------------------------------------------------------------------------------ */
/* Loss scaler and step counter.                                                        */
/* ------------------------------------------------------------------------------------ */

/* [ZO] config: fp16 training is enabled, which implies loss scaling with overflow
 * handling; the policy is not on the pages.  Reading: on overflow the step is skipped
 * (no state changes, t unchanged), a dynamic scale halves (floor 1) and the good-step
 * count restarts; otherwise t advances and, for a dynamic scale, every G-th consecutive
 * good step doubles L (cap 2^24).  A static scale (bf16 training) never changes. */
int oracle_scaler_update(oracle_scaler_t* s, uint32_t overflow)
{
    if (overflow) {
        if (s->dynamic) {
            float half = s->loss_scale * 0.5f;
            s->loss_scale = half < 1.0f ? 1.0f : half;
            s->good_steps = 0;
        }
        s->n_skipped += 1;
        return 0;
    }
    s->t += 1;
    if (s->dynamic && s->growth_interval > 0) {
        s->good_steps += 1;
        if (s->good_steps == s->growth_interval) {
            float twice = s->loss_scale * 2.0f;
            s->loss_scale = twice > 16777216.0f ? 16777216.0f : twice;
            s->good_steps = 0;
        }
    }
    return 1;
}

/* ------------------------------------------------------------------------------------ */
/* AdamW on the fp32 master / momentum / variance shard, bf16 cast.                      */
/* ------------------------------------------------------------------------------------ */

/* Bias corrections of Adam (Kingma & Ba, 2015) for step t, in fp64, rounded once:
 * step_size = lr / (1 - beta1^t), rbc2 = sqrt(1 - beta2^t), and the decoupled weight-decay
 * factor 1 - lr*wd (Loshchilov & Hutter, 2019). */
void oracle_adamw_scalars(const oracle_hparams_t* hp, uint32_t t, float* step_size,
                          float* rbc2, float* decay)
{
    double bc1 = 1.0 - pow((double)hp->beta1, (double)t);
    double bc2 = 1.0 - pow((double)hp->beta2, (double)t);
    *step_size = (float)((double)hp->lr / bc1);
    *rbc2 = (float)sqrt(bc2);
    *decay = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);
}

/* [ZW] sec. 6(2): each GPU runs the optimizer on its own parameters with its own reduced
 * gradient; [ZS] and [MD] name the optimizer AdamW but do not write it.  Reading: Adam
 * with bias correction and decoupled weight decay, one element at a time in fp32:
 *   gc = c*g;  m = b1*m + (1-b1)*gc;  v = b2*v + (1-b2)*(gc*gc)
 *   p  = p*(1 - lr*wd) - step_size * (m / (sqrt(v)/rbc2 + eps))
 * and the fp32 master is cast to bf16 with round-to-nearest-even (or, as a variant, to
 * fp16: [ZW] sec. 4(1) keeps the replicated parameters in FP16). */
static uint16_t adamw_one(const oracle_hparams_t* hp, float c, float step_size, float rbc2,
                          float decay, float g, float* p, float* m, float* v)
{
    float b1 = hp->beta1;
    float b2 = hp->beta2;
    float omb1 = 1.0f - b1;
    float omb2 = 1.0f - b2;
    float gc = c * g;
    float m_new = b1 * *m + omb1 * gc;
    float v_new = b2 * *v + omb2 * (gc * gc);
    float denom = sqrtf(v_new) / rbc2 + hp->eps;
    float p_new = *p * decay - step_size * (m_new / denom);
    *m = m_new;
    *v = v_new;
    *p = p_new;
    return hp->params_dtype == ORACLE_F16 ? oracle_f32_to_f16(p_new) : oracle_f32_to_bf16(p_new);
}

void oracle_adamw_elements(const oracle_hparams_t* hp, float clip_coef, uint32_t t, uint64_t n,
                           const float* g, float* master, float* m, float* v, uint16_t* out)
{
    float step_size, rbc2, decay;
    oracle_adamw_scalars(hp, t, &step_size, &rbc2, &decay);
    for (uint64_t i = 0; i < n; ++i)
        out[i] = adamw_one(hp, clip_coef, step_size, rbc2, decay, g[i], &master[i], &m[i], &v[i]);
}

/* [ZW] sec. 4(1) and 6(2): rank r updates only partition r, and the all-gather that
 * follows rebuilds the full parameter vector [p0' ... p7'] with every shard at its own
 * offset; writing rank r's bf16 result at flat offsets [r*S, (r+1)*S) of one buffer is
 * that gathered layout.  [ZS]: the gathered weights are bf16. */
void oracle_adamw_shard(const oracle_layout_t* lay, const oracle_hparams_t* hp, float clip_coef,
                        uint32_t t, uint64_t rank, const float* g, float* master, float* m,
                        float* v, uint16_t* out)
{
    float step_size, rbc2, decay;
    oracle_adamw_scalars(hp, t, &step_size, &rbc2, &decay);
    uint64_t lo = rank * lay->shard;
    uint64_t hi = lo + lay->shard;
    for (uint64_t i = lo; i < hi; ++i) {
        if (i >= lay->psi) {
            out[i] = 0;  /* padding: gathered value 0, state untouched */
            continue;
        }
        out[i] = adamw_one(hp, clip_coef, step_size, rbc2, decay, g[i], &master[i], &m[i], &v[i]);
    }
}

/* ------------------------------------------------------------------------------------ */
/* Whole steps.                                                                         */
/* ------------------------------------------------------------------------------------ */

/* One iteration's optimizer part in the order of [ZO] "method flow" (stage 2): gradient
 * reduce-scatter, optimizer update of each shard, parameter all-gather, with the global
 * norm all-reduce of [MD] sec. 1 before clipping and the overflow skip of fp16 training.
 * The stage only changes which buffers persist (the ledger), not this arithmetic. */
int oracle_step(const oracle_layout_t* lay, const oracle_hparams_t* hp, int dtype,
                const uint16_t* const* replicas, float* g, float* master, float* m, float* v,
                uint16_t* out, oracle_scaler_t* sc, oracle_report_t* rep)
{
    uint64_t N = lay->n_ranks;
    uint64_t S = lay->shard;
    if (dtype != ORACLE_F16 && dtype != ORACLE_BF16)
        return -1;
    double* sumsq = (double*)calloc(N, sizeof(double));
    const uint16_t** shard_ptrs = (const uint16_t**)malloc(N * sizeof(*shard_ptrs));
    if (!sumsq || !shard_ptrs) {
        free(sumsq);
        free(shard_ptrs);
        return -1;
    }
    float inv = oracle_inv_scale(N, sc->loss_scale);
    uint32_t overflow = 0;

    /* reduce-scatter: rank r receives the average of every rank's copy of shard r */
    for (uint64_t r = 0; r < N; ++r) {
        for (uint64_t k = 0; k < N; ++k)
            shard_ptrs[k] = replicas[k] + r * S;
        oracle_reduce_window(lay, dtype, shard_ptrs, r * S, S, inv, g + r * S, sumsq, &overflow);
    }

    double total;
    double norm = oracle_global_norm(sumsq, N, &total);
    float used = sc->loss_scale;
    int applied = oracle_scaler_update(sc, overflow);
    float c = applied ? oracle_clip_coef(norm, hp->max_grad_norm) : 1.0f;
    if (applied)
        for (uint64_t r = 0; r < N; ++r)
            oracle_adamw_shard(lay, hp, c, sc->t, r, g, master, m, v, out);

    if (rep) {
        rep->sumsq = total;
        rep->norm = norm;
        rep->clip_coef = c;
        rep->loss_scale_used = used;
        rep->loss_scale_next = sc->loss_scale;
        rep->overflow = overflow;
        rep->skipped = !applied;
        rep->t = sc->t;
    }
    free(sumsq);
    free(shard_ptrs);
    return 0;
}

/* Plain data parallelism after the all-reduce: every rank holds the averaged gradient
 * and updates all Psi parameters.  [ZS] calls ZeRO-1 exactly this all-reduce, split in
 * two; the sharded step must give the same numbers. */
int oracle_step_unsharded(uint64_t psi, const oracle_hparams_t* hp, const float* g_mean,
                          float* master, float* m, float* v, uint16_t* out, oracle_scaler_t* sc,
                          oracle_report_t* rep)
{
    double q = 0.0;
    uint32_t overflow = 0;
    for (uint64_t i = 0; i < psi; ++i) {
        if (!isfinite(g_mean[i]))
            overflow = 1;
        q = q + (double)g_mean[i] * (double)g_mean[i];
    }
    double norm = sqrt(q);
    float used = sc->loss_scale;
    int applied = oracle_scaler_update(sc, overflow);
    float c = applied ? oracle_clip_coef(norm, hp->max_grad_norm) : 1.0f;
    if (applied)
        oracle_adamw_elements(hp, c, sc->t, psi, g_mean, master, m, v, out);
    if (rep) {
        rep->sumsq = q;
        rep->norm = norm;
        rep->clip_coef = c;
        rep->loss_scale_used = used;
        rep->loss_scale_next = sc->loss_scale;
        rep->overflow = overflow;
        rep->skipped = !applied;
        rep->t = sc->t;
    }
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Per-tensor segment map.                                                               */
/* [ZW] sec. 4(2): gradients are bucketed by partition and each bucket is reduced at the */
/* partition boundary, so a tensor that crosses a boundary is split between two owners. */
/* Brute force, one flat element at a time.                                              */
/* ------------------------------------------------------------------------------------ */

int64_t oracle_segment_map(const oracle_layout_t* lay, const uint64_t* tensor_elems,
                           uint64_t n_tensors, oracle_segment_t* out, uint64_t capacity)
{
    uint64_t total = 0;
    for (uint64_t k = 0; k < n_tensors; ++k)
        total += tensor_elems[k];
    if (total != lay->psi)
        return -1;
    int64_t n = 0;
    uint64_t k = 0, start_of_k = 0;   /* tensor k covers flat [start_of_k, start_of_k + size) */
    uint64_t cur_tensor = UINT64_MAX, cur_rank = UINT64_MAX;
    for (uint64_t i = 0; i < lay->psi; ++i) {
        while (i >= start_of_k + tensor_elems[k]) {   /* skips empty tensors too */
            start_of_k += tensor_elems[k];
            ++k;
        }
        uint64_t r = i / lay->shard;
        if (k != cur_tensor || r != cur_rank) {
            cur_tensor = k;
            cur_rank = r;
            if ((uint64_t)n < capacity) {
                out[n].tensor = k;
                out[n].rank = r;
                out[n].tensor_offset = i - start_of_k;
                out[n].shard_offset = i - r * lay->shard;
                out[n].count = 0;
            }
            ++n;
        }
        if ((uint64_t)(n - 1) < capacity)
            out[n - 1].count += 1;
    }
    return n;
}

