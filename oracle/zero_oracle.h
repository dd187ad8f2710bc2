/*
 * zero_oracle.h -- CPU oracle for the ZeRO-DP partitioned mixed-precision AdamW step.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load this library.  It shares no code
 * with the CUDA library: its own number-format conversions, its own layout arithmetic,
 * its own loops.
 *
 * Everything here is plain serial C compiled with -O2 -ffp-contract=off (no fused
 * multiply-add, no fast-math), so each floating-point operation is exactly the one written.
 *
 * Sources (web pages on ZeRO):
 *   [ZW] "【论文解读】ZeRO", wkq9411.github.io (a walkthrough of the ZeRO paper)
 *   [ZM] "ZeRO 显存优化：ZeRO-1、ZeRO-2 与 ZeRO-3", xiangdong0520.pages.dev
 *   [ZS] "ZeRO optimizer sharding", operatorworld.com/p/ai/ai-zero-optimizer-sharding
 *   [ZO] "3、ZeRO技术概述：ZeRO三个阶段原理与对比", 5688vip.com (DeepSpeed chapter)
 *   [MD] "Megatron distributed optimizer and ZeRO", gitcode.csdn.net/69f2000254b52172bc70cc37
 *
 * The parity pins of each function (tests/test_oracle_*.py) are listed in zero_oracle.c;
 * no function is left without one.
 */
#ifndef ZERO_ORACLE_H
#define ZERO_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_F16 1
#define ORACLE_BF16 2

/* Partition of Psi flat parameters into N equal padded shards, with the model-state
 * ledger and the per-rank communication volume for plain DP (stage 0) and stages 1-3. */
typedef struct oracle_layout {
    uint64_t psi;              /* parameters */
    uint64_t n_ranks;          /* N_d */
    uint64_t shard;            /* S: elements per rank */
    uint64_t psi_padded;       /* N * S */
    uint64_t pad;              /* N * S - Psi */
    uint64_t align;            /* S is a multiple of align */
    uint64_t bucket_elems;     /* bucket (window) size W over the flat index */
    uint64_t n_buckets;        /* ceil(psi_padded / W) */
    uint64_t stage;            /* 0 = plain DP, 1 = P_os, 2 = P_os+g, 3 = P_os+g+p */
    uint64_t bytes_per_rank[4];      /* model-state bytes held by one rank, per stage */
    uint64_t comm_elems_per_rank[4]; /* elements one rank sends per step, per stage */
} oracle_layout_t;

typedef struct oracle_hparams {
    float lr, beta1, beta2, eps, weight_decay, max_grad_norm;
    uint32_t params_dtype;     /* gathered parameters: 0 or ORACLE_BF16 = bf16, ORACLE_F16 = fp16 */
} oracle_hparams_t;

/* Loss scaler and step counter. */
typedef struct oracle_scaler {
    float loss_scale;          /* L used to generate (and to divide out of) the gradients */
    uint32_t dynamic;          /* 1: back off / grow L; 0: L is static */
    uint32_t growth_interval;  /* G: good steps between doublings (0 = never grow) */
    uint32_t good_steps;
    uint32_t t;                /* applied optimizer steps */
    uint32_t n_skipped;
} oracle_scaler_t;

/* What one step produced. */
typedef struct oracle_report {
    double sumsq;              /* sum of g^2 over all ranks (fp64) */
    double norm;               /* sqrt(sumsq) */
    float clip_coef;           /* c actually applied (1 when skipped) */
    float loss_scale_used;     /* L of this step's gradients */
    float loss_scale_next;     /* L after the scaler update */
    uint32_t overflow;         /* any non-finite reduced gradient */
    uint32_t skipped;          /* step skipped because of overflow */
    uint32_t t;                /* step counter after this step */
} oracle_report_t;

/* number formats */
float oracle_f16_to_f32(uint16_t h);
float oracle_bf16_to_f32(uint16_t b);
uint16_t oracle_f32_to_bf16(float x);
uint16_t oracle_f32_to_f16(float x);

/* layout and ledger; returns 0 or -1 on invalid arguments */
int oracle_partition(uint64_t psi, uint64_t n_ranks, uint32_t stage, uint64_t align,
                     uint64_t bucket_elems, oracle_layout_t* out);

/* f32(1 / (N * L)) */
float oracle_inv_scale(uint64_t n_ranks, float loss_scale);

/* Reduce-scatter arithmetic over the flat window [begin, begin+count).
 * replicas[k] points at flat element `begin` of rank k's gradient (bit patterns of
 * dtype ORACLE_F16 / ORACLE_BF16); g also points at flat element `begin` and receives
 * count fp32 values.  Adds each element's g^2 to sumsq[owner rank] (sumsq has n_ranks
 * entries, indexed by rank) and ORs the overflow flag. */
void oracle_reduce_window(const oracle_layout_t* lay, int dtype, const uint16_t* const* replicas,
                          uint64_t begin, uint64_t count, float inv_scale, float* g,
                          double* sumsq, uint32_t* overflow);

/* sqrt of the rank-ordered sum of the per-rank sums of squares */
double oracle_global_norm(const double* sumsq, uint64_t n_ranks, double* total);

/* c = min(1, max_norm / (norm + 1e-6)); 1 when max_norm <= 0 */
float oracle_clip_coef(double norm, float max_norm);

/* Scaler policy; returns 1 when the step is applied (t advanced), 0 when skipped. */
int oracle_scaler_update(oracle_scaler_t* s, uint32_t overflow);

/* Per-step AdamW scalars for step t >= 1. */
void oracle_adamw_scalars(const oracle_hparams_t* hp, uint32_t t, float* step_size,
                          float* rbc2, float* decay);

/* AdamW on n independent elements (no padding rule); writes the gathered parameters'
 * bit patterns (bf16, or fp16 when hp->params_dtype == ORACLE_F16) to out. */
void oracle_adamw_elements(const oracle_hparams_t* hp, float clip_coef, uint32_t t, uint64_t n,
                           const float* g, float* master, float* m, float* v, uint16_t* out);

/* AdamW on rank r's shard [r*S, (r+1)*S) of the flat arrays, writing the bf16 result at
 * the same flat offsets of the gathered parameter buffer.  Pad positions (>= psi) get
 * out = 0 and their master/m/v are left untouched. */
void oracle_adamw_shard(const oracle_layout_t* lay, const oracle_hparams_t* hp, float clip_coef,
                        uint32_t t, uint64_t rank, const float* g, float* master, float* m,
                        float* v, uint16_t* out);

/* One whole sharded step: reduce-scatter of every rank's shard, global norm, scaler,
 * clip, AdamW per shard, bf16 gather.  replicas[k] covers the full flat buffer
 * [0, psi_padded).  Returns 0, or -1 on invalid arguments. */
int oracle_step(const oracle_layout_t* lay, const oracle_hparams_t* hp, int dtype,
                const uint16_t* const* replicas, float* g, float* master, float* m, float* v,
                uint16_t* out, oracle_scaler_t* sc, oracle_report_t* rep);

/* The unsharded step on an already averaged and unscaled fp32 gradient of psi elements
 * (plain data parallelism after the all-reduce).  Same scaler, clip and AdamW. */
int oracle_step_unsharded(uint64_t psi, const oracle_hparams_t* hp, const float* g_mean,
                          float* master, float* m, float* v, uint16_t* out, oracle_scaler_t* sc,
                          oracle_report_t* rep);

/* One piece of a model tensor inside one rank's shard. */
typedef struct oracle_segment {
    uint64_t tensor;           /* index in the tensor list */
    uint64_t rank;             /* owner of the piece */
    uint64_t tensor_offset;    /* first element of the piece within the tensor */
    uint64_t shard_offset;     /* the same element's position within the owner's shard */
    uint64_t count;            /* elements in the piece */
} oracle_segment_t;

/* Tensors of the given sizes laid end to end over the flat buffer [0, psi), in list
 * order, cut at the shard boundaries: walks every flat element and starts a new piece
 * whenever the (tensor, rank) pair changes.  Writes at most `capacity` pieces in flat
 * order and returns how many there are, or -1 if the sizes do not sum to psi. */
int64_t oracle_segment_map(const oracle_layout_t* lay, const uint64_t* tensor_elems,
                           uint64_t n_tensors, oracle_segment_t* out, uint64_t capacity);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_ORACLE_H */
