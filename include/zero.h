/*
 * zero.h -- C ABI of the GB300 (sm_103a) ZeRO-DP partitioned mixed-precision AdamW step.
 *
 * One optimizer step of ZeRO-DP data parallelism with all N data-parallel ranks held as
 * buffers on one GPU (or, through the rank-local entry points, spread over processes):
 *   1. partition      Psi flat parameters into N equal, padded shards (rank r owns
 *                     flat [r*S, (r+1)*S)), with the per-rank model-state ledger
 *   2. reduce-scatter average the N ranks' fp16/bf16 gradient copies into fp32, remove
 *                     the loss scale, flag inf/NaN, and sum g^2 per tile of a shard
 *   3. grad norm      global L2 norm of the averaged gradient, clip coefficient,
 *                     loss-scale update and the skip decision, all on the device
 *   4. AdamW + cast   update the fp32 master / momentum / variance of every shard and
 *                     write each shard's bf16 parameters at its own offset r*S of one
 *                     gathered buffer (the layout the parameter all-gather produces);
 *                     the state may also live in host memory
 * plus the per-tensor segment map (which rank owns which piece of each model tensor).
 * zero_step runs steps 2-4 as one kernel per part (a reduce per gradient bucket, the
 * norm, AdamW) on large layouts and as ONE cooperative kernel, with the same bits, on
 * small ones (zero_step_launches).
 *
 * Sources (web pages on ZeRO):
 *   [ZW] "【论文解读】ZeRO", wkq9411.github.io: sec. 4(1)-(3) the three partitioning stages,
 *        sec. 6(1)-(2) reduce-scatter / all-gather and the 8-parameter, 4-GPU example
 *   [ZM] "ZeRO 显存优化：ZeRO-1、ZeRO-2 与 ZeRO-3", xiangdong0520.pages.dev: sec. 2-3 ledger,
 *        sec. 6 optimizer state offloaded to the CPU
 *   [ZS] operatorworld.com ZeRO optimizer-sharding article: AdamW 16-byte ledger (bf16
 *        weights and gradients), stage flows, communication accounting
 *   [ZO] "3、ZeRO技术概述：ZeRO三个阶段原理与对比", 5688vip.com: stage-2 iteration flow,
 *        DeepSpeed config with "fp16": enabled
 *   [MD] gitcode.csdn.net article on Megatron's distributed optimizer: sec. 1 global
 *        grad-norm all-reduce before clip_coeff
 *
 * Conventions for every function below:
 *   - Ownership: the caller allocates and frees every buffer.  No function allocates or
 *     frees device memory; zero_step_host creates and destroys four CUDA events.
 *   - Device pointers must be 16-byte aligned (ZERO_EALIGN otherwise).
 *   - Asynchrony: device work is enqueued on the caller's stream and the call returns
 *     without waiting, except zero_step_state_read / zero_step_state_write, which wait.
 *   - Errors: arguments are validated on the host before anything is enqueued; a
 *     rejected call changes nothing.  A launch failure returns ZERO_ECUDA and
 *     zero_last_cuda_error() gives the CUDA error code.  Faults inside kernels surface at
 *     the caller's next synchronisation.  Overflow of the gradients is not an error: it
 *     is reported in the step state and the step is skipped.
 *   - Thread safety: calls on different streams may run concurrently if they share no
 *     buffers.
 *   - Profiling: every device entry point opens an NVTX range named after itself.
 */
#ifndef ZERO_H
#define ZERO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* zero_stream_t;

#define ZERO_OK 0
#define ZERO_EINVAL (-1)   /* invalid argument */
#define ZERO_EALIGN (-2)   /* pointer or window not aligned as required */
#define ZERO_ENOMEM (-3)   /* caller-provided buffer too small */
#define ZERO_ECUDA (-4)    /* CUDA launch or copy failed; see zero_last_cuda_error() */
#define ZERO_ETIMEOUT (-5) /* reserved; a device wait that gives up records 1 in the step
                              state's error word instead */

typedef enum zero_dtype { ZERO_F16 = 1, ZERO_BF16 = 2 } zero_dtype_t;

#define ZERO_MAX_RANKS (1u << 20)   /* zero_partition (ledger and layout) */
#define ZERO_MAX_KERNEL_RANKS 64u   /* device entry points: replicas summed per element */
#define ZERO_TILE_ELEMS 8192u       /* grid of the sum-of-squares partials' tiles */

/* Partition of Psi flat parameters over N ranks.  Filled by zero_partition; pass it back
 * unchanged to the device entry points (they re-check its invariants). */
typedef struct zero_layout {
    uint64_t psi;                    /* Psi: parameters */
    uint64_t shard;                  /* S = ceil(Psi/N) rounded up to align: elements per rank */
    uint64_t psi_padded;             /* N*S: length of every flat buffer */
    uint64_t pad;                    /* N*S - Psi: trailing padding, gradient 0, output 0 */
    uint64_t bucket_elems;           /* W: window of one reduce launch in zero_step */
    uint64_t n_buckets;              /* ceil(N*S / W) */
    uint64_t tiles_per_rank;         /* ceil(S / tile_elems) + 1: a shard meets at most this
                                        many cells of the flat tile grid */
    uint64_t n_tiles;                /* N * tiles_per_rank: fp64 partial slots */
    uint64_t bytes_per_rank[4];      /* model-state bytes per rank: [0] plain DP 16*Psi,
                                        [1] 4*N*S + 12*S, [2] 2*N*S + 14*S, [3] 16*S */
    uint64_t comm_elems_per_rank[4]; /* elements each rank sends per step on a ring:
                                        2(N-1)S for [0..2], 3(N-1)S for stage 3 */
    uint32_t n_ranks;                /* N */
    uint32_t stage;                  /* 0 plain DP, 1 P_os, 2 P_os+g, 3 P_os+g+p */
    uint32_t align;                  /* S is a multiple of align */
    uint32_t tile_elems;             /* ZERO_TILE_ELEMS */
} zero_layout_t;

typedef struct zero_adamw_hparams {
    float lr;
    float beta1;            /* in [0, 1) */
    float beta2;            /* in [0, 1) */
    float eps;              /* > 0 */
    float weight_decay;     /* decoupled: p *= 1 - lr*weight_decay */
    float max_grad_norm;    /* global-norm clip threshold; <= 0 disables clipping */
    uint32_t params_dtype;  /* gathered parameters: 0 or ZERO_BF16 = bf16 (the default);
                               ZERO_F16 = fp16, the FP16 replicated parameters of
                               "【论文解读】ZeRO" sec. 4(1) */
} zero_adamw_hparams_t;

/* Scalar step state.  Lives in DEVICE memory (caller allocates sizeof(zero_step_state_t)
 * bytes, 16-byte aligned); read it with zero_step_state_read. */
typedef struct zero_step_state {
    double sumsq;           /* sum of g^2 of the last finalised step (fp64) */
    double norm;            /* its square root: the global L2 gradient norm */
    float clip_coef;        /* c applied by the last finalised step (1 when skipped) */
    float loss_scale;       /* L of the NEXT step's gradients */
    float inv_scale;        /* f32(1 / (N*L)): the reduce's unscale factor */
    float step_size;        /* lr / (1 - beta1^t) for the step being applied */
    float rbc2;             /* sqrt(1 - beta2^t) */
    float decay;            /* 1 - lr*weight_decay */
    uint32_t overflow;      /* non-finite seen by this step's reduce windows so far */
    uint32_t skip;          /* 1 if the last finalised step was skipped (overflow) */
    uint32_t t;             /* applied optimizer steps */
    uint32_t good_steps;    /* consecutive applied steps since the last scale change */
    uint32_t growth_interval;
    uint32_t dynamic;       /* 1: dynamic loss scale (halve on overflow, double every
                               growth_interval good steps, floor 1, cap 2^24) */
    uint32_t n_ranks;
    uint32_t n_steps;       /* finalised steps, applied or skipped */
    uint32_t n_skipped;
    uint32_t error;         /* device error word: 0 = none; 1 = a bounded wait gave up;
                               2 = (checked test builds only) a store outside its range */
    uint32_t arrivals;      /* internal to zero_grad_norm: its blocks that have finished
                               (0 between steps; keep it 0 when writing a state) */
    float inv_scale_used;   /* the inv_scale the last finalised step's reduce used */
    uint32_t launch_arrivals; /* internal to zero_step's single launch: its blocks that
                               have finished their reduce (0 between steps; keep it 0
                               when writing a state) */
    float applied_c;        /* the clip coefficient the last finalised step applied, -1
                               when it was skipped, 0 before the first step; the single
                               launch hands it to its blocks together with
                               launch_arrivals in one 64-bit store */
    uint64_t adamw_next_chunk; /* internal to the AdamW pass: the next chunk its blocks
                               take (0 between steps; keep it 0 when writing a state) */
    uint32_t adamw_done;    /* internal to the AdamW pass: its blocks that have finished;
                               the last one puts both words back to 0 */
    uint32_t reserved[5];
} zero_step_state_t;        /* 128 bytes */

/* -------------------------------------------------------------------------------------
 * zero_partition -- host only, no CUDA call.
 * [ZW] sec. 4(1)-(3): N equal partitions, rank r owns partition r; the ledger per stage
 * ([ZW] sec. 2(1) and 8, [ZM] sec. 3): 16*Psi, (4 + 12/N)Psi, (2 + 14/N)Psi, 16*Psi/N,
 * counted on the padded buffers; the ring traffic of [ZW] sec. 6 eq. dp-comm.
 *   psi           >= 1, <= 2^56
 *   n_ranks       1 .. ZERO_MAX_RANKS
 *   stage         0 .. 3 (0 = plain data parallelism, for the ledger only)
 *   align         S is rounded up to a multiple of align (1 .. 2^20)
 *   bucket_elems  window of one reduce launch in zero_step; 0, or any value of at least
 *                 N*S, = one window over the whole flat buffer; otherwise a multiple of 8
 *   out           written on success
 * Returns ZERO_OK or ZERO_EINVAL.
 * ------------------------------------------------------------------------------------- */
int zero_partition(uint64_t psi, uint32_t n_ranks, uint32_t stage, uint32_t align,
                   uint64_t bucket_elems, zero_layout_t* out);

/* One piece of a model tensor inside one rank's shard. */
typedef struct zero_segment {
    uint64_t tensor;         /* index in the caller's tensor list */
    uint64_t rank;           /* owner of the piece */
    uint64_t tensor_offset;  /* first element of the piece within the tensor */
    uint64_t shard_offset;   /* the same element's position in the owner's shard
                                (flat index - rank*S) */
    uint64_t count;          /* elements in the piece (>= 1) */
} zero_segment_t;            /* 40 bytes */

/* -------------------------------------------------------------------------------------
 * zero_segment_map -- host only, no CUDA call.
 * [ZW] sec. 4(2): gradients are bucketed by partition and reduced at the partition
 * boundary, so a tensor that crosses a shard boundary belongs to two or more ranks.
 * The model's tensors are laid end to end over the flat buffer [0, psi) in list order;
 * this lists each tensor's piece on each rank, in flat order (so by rank, then tensor).
 * Empty tensors have no piece; padding [psi, psi_padded) belongs to no tensor.
 *   tensor_elems   HOST array of n_tensors element counts; they must sum to layout->psi
 *   out            HOST array of `capacity` pieces, or NULL to only count them
 *   n_segments     HOST, receives the number of pieces (always, on ZERO_OK or ZERO_ENOMEM)
 * Returns ZERO_OK; ZERO_EINVAL (bad layout or pointers, sizes not summing to psi);
 * ZERO_ENOMEM when capacity is too small (out untouched).  There are
 * (non-empty tensors) + (shard boundaries strictly inside a tensor) pieces.
 * ------------------------------------------------------------------------------------- */
int zero_segment_map(const zero_layout_t* layout, const uint64_t* tensor_elems,
                     uint64_t n_tensors, zero_segment_t* out, uint64_t capacity,
                     uint64_t* n_segments);

/* Bytes of the fp64 partials workspace the device entry points need:
 * layout->n_tiles * 8.  0 for an invalid layout. */
size_t zero_workspace_bytes(const zero_layout_t* layout);

/* -------------------------------------------------------------------------------------
 * zero_step_state_init -- start a fresh optimizer (t = 0) on the device.
 *   loss_scale       initial L (> 0, finite); 1 for bf16 training
 *   dynamic          1: dynamic loss scaling (fp16 training, [ZO] "fp16": enabled);
 *                    0: static scale, overflow still skips the step
 *   growth_interval  good steps between doublings of a dynamic scale (0 = never)
 *   st               device, sizeof(zero_step_state_t)
 *   partials         device, zero_workspace_bytes(layout); zeroed here
 * Enqueues one kernel on `stream`.
 * ------------------------------------------------------------------------------------- */
int zero_step_state_init(const zero_layout_t* layout, float loss_scale, uint32_t dynamic,
                         uint32_t growth_interval, zero_step_state_t* st, double* partials,
                         zero_stream_t stream);

/* Copy the device state to host memory and wait for it (checkpoints, monitoring). */
int zero_step_state_read(const zero_step_state_t* st, zero_step_state_t* host_out,
                         zero_stream_t stream);

/* Copy a host state (e.g. from a checkpoint) to the device and wait for it.  The
 * kernels' internal counters (arrivals, launch_arrivals, adamw_next_chunk, adamw_done)
 * are written as 0 whatever host_in holds. */
int zero_step_state_write(zero_step_state_t* st, const zero_step_state_t* host_in,
                          zero_stream_t stream);

/* -------------------------------------------------------------------------------------
 * zero_reduce_shard_unscale -- the reduce-scatter arithmetic on one flat window.
 * [ZW] sec. 6(1)-(2): the ranks' gradients are averaged; with gradient partitioning the
 * average is reduce-scattered so rank r receives only flat [r*S, (r+1)*S).  [ZW] sec. 4(2):
 * gradients are bucketed and each bucket reduced as it becomes ready.
 * For every flat i in [begin, begin+count):
 *   g[i] = (sum over k = 0..N-1, ascending, in fp32, of x_k[i]) * st->inv_scale
 *   with g[i] = 0 for padding (i >= psi; replica values there are ignored);
 *   st->overflow |= any non-finite g[i];
 *   partials[tile of i] += sum of g^2 over the window's part of each tile.  Tiles cut
 *   each shard at the flat multiples of T = tile_elems (so interior tiles start on
 *   128-byte lines of every array): tile j of rank r is the intersection of
 *   [r*S, (r+1)*S) with [(c+j)*T, (c+j+1)*T), c = floor(r*S/T); slot r*tiles_per_rank + j.
 *   A rank's trailing slots may be empty (always 0).
 *   dtype      ZERO_F16 or ZERO_BF16 (the replicas' element type)
 *   replicas   HOST array of N DEVICE pointers; replicas[k] points at flat element
 *              `begin` of rank k's gradient copy and holds at least `count` elements
 *   begin      multiple of 8 (ZERO_EALIGN otherwise); begin + count <= psi_padded
 *   g          DEVICE fp32 array of psi_padded elements (indexed by the flat index)
 *   partials   DEVICE, zero_workspace_bytes(layout); zeroed by zero_step_state_init and
 *              by every zero_grad_norm, accumulated here
 *   st         DEVICE step state
 * N must be <= ZERO_MAX_KERNEL_RANKS.  Windows of one step may come in any order but
 * must not overlap; together they must cover [0, psi_padded) before zero_grad_norm.
 * ------------------------------------------------------------------------------------- */
int zero_reduce_shard_unscale(const zero_layout_t* layout, zero_dtype_t dtype,
                              const void* const* replicas, uint64_t begin, uint64_t count,
                              float* g, double* partials, zero_step_state_t* st,
                              zero_stream_t stream);

/* -------------------------------------------------------------------------------------
 * zero_grad_norm -- global norm, clip coefficient, loss scaler and skip decision.
 * [MD] sec. 1: inside optimizer.step(), before clipping, one all-reduce forms the global
 * L2 gradient norm that sets clip_coeff.  Here the all-reduce is the fixed-order sum of
 * the per-rank partial sums (each rank's tiles, then ranks in order):
 *   norm = sqrt(sumsq);  c = min(1, max_norm / (norm + 1e-6)) (fp64, rounded to fp32)
 *   overflow: skip = 1, c = 1, t unchanged, dynamic L = max(L/2, 1)
 *   else:     skip = 0, t += 1, step_size = f32(lr/(1-beta1^t)), rbc2 = f32(sqrt(1-beta2^t)),
 *             decay = f32(1 - lr*wd); dynamic L doubles after growth_interval good steps
 *   inv_scale = f32(1/(N*L)) for the next step; overflow flag and partials reset to 0.
 * One kernel (the partial sums spread over up to 128 blocks, the last block to finish
 * forms the norm); no host synchronisation.
 * ------------------------------------------------------------------------------------- */
int zero_grad_norm(const zero_layout_t* layout, const zero_adamw_hparams_t* hp,
                   double* partials, zero_step_state_t* st, zero_stream_t stream);

/* -------------------------------------------------------------------------------------
 * zero_adamw_cast_gather -- fused AdamW on every shard plus the gathered write (bf16, or
 * fp16 when hp->params_dtype == ZERO_F16).
 * [ZW] sec. 6(2): each rank updates its own parameters from its own reduced gradient and
 * the all-gather rebuilds [p0' ... p7'] in order; [ZS]: AdamW, bf16 weights.
 * Does nothing (on the device) when st->skip.  Otherwise, per flat i < psi, in fp32:
 *   gc = c*g;  m = b1*m + (1-b1)*gc;  v = b2*v + (1-b2)*(gc*gc)
 *   p  = p*decay - step_size * (m / (sqrt(v)/rbc2 + eps));  params[i] = bf16_rne(p)
 * and params[i] = 0 for padding (master/m/v there untouched).
 *   g, master, m, v   DEVICE fp32, psi_padded elements each (master/m/v updated in place)
 *   params            DEVICE bf16 (or fp16) bit patterns (uint16), psi_padded elements
 *   hp                must equal the hp given to zero_grad_norm for this step
 * ------------------------------------------------------------------------------------- */
int zero_adamw_cast_gather(const zero_layout_t* layout, const zero_adamw_hparams_t* hp,
                           const float* g, float* master, float* m, float* v, uint16_t* params,
                           const zero_step_state_t* st, zero_stream_t stream);

/* -------------------------------------------------------------------------------------
 * zero_adamw_cast_gather_host_state -- zero_adamw_cast_gather with the optimizer state
 * (master, m, v) resident in HOST memory.
 * [ZM] sec. 6: when device memory is short the optimizer state can be offloaded to the
 * CPU, at a transfer cost that has to be measured on the machine.  Here the state stays
 * in the host memory of the Grace CPU and the kernel reads and writes it in place over
 * the CPU-GPU link (NVLink-C2C on GB300) while g is read from, and the gathered
 * parameters written to, device memory; 12 B per element cross the link each way.
 * Same update, same bits as zero_adamw_cast_gather.
 *   master, m, v   HOST fp32, psi_padded elements each, PAGE-LOCKED (cudaHostAlloc /
 *                  cudaMallocHost / cudaHostRegister, e.g. torch pin_memory); updated in
 *                  place.  Pageable or device memory is refused with ZERO_EINVAL.  The
 *                  host must not touch them until the stream has passed this call.
 *   g, params, st  DEVICE, as in zero_adamw_cast_gather
 * ------------------------------------------------------------------------------------- */
int zero_adamw_cast_gather_host_state(const zero_layout_t* layout,
                                      const zero_adamw_hparams_t* hp, const float* g,
                                      float* master, float* m, float* v, uint16_t* params,
                                      const zero_step_state_t* st, zero_stream_t stream);

/* -------------------------------------------------------------------------------------
 * Rank-local entry points: the step with the ranks spread over processes (one process per
 * GPU), each process holding only its own ranks' part of g and of the optimizer state.
 * [ZW] sec. 6(2) and [ZO] stage-2 flow: each rank receives every rank's gradient for its
 * own partition (reduce-scatter), updates only its partition, and the updated parameters
 * are all-gathered; [MD] sec. 1: the global norm needs one all-reduce before clipping.
 *
 * A process holds the contiguous ranks [rank_begin, rank_begin + rank_count) (one rank per
 * process, or several); their flat range starts at origin = rank_begin*S and is
 * local_len = rank_count*S long.  Local buffers are indexed by flat index - origin.
 * origin must be a multiple of 8 (partition with align = 8; ZERO_EALIGN otherwise).
 * One step, per process, with the exchanges done by the caller (e.g. NCCL):
 *   1. exchange: every rank's gradient copy of the local range arrives (rank k's copy of
 *      flat [origin, origin + local_len)), whole or window by window (an all-to-all, or
 *      point-to-point sends of each window);
 *   2. zero_reduce_shard_unscale_local over the local range (one or more windows; the
 *      result does not depend on the windows when their boundaries lie on the flat
 *      multiples of ZERO_TILE_ELEMS);
 *   3. exchange: all-gather every process's partial slots [rank_begin*tiles_per_rank,
 *      (rank_begin + rank_count)*tiles_per_rank) into the full partials array, and
 *      combine the step state's `overflow` word over processes (maximum);
 *   4. zero_grad_norm on the full partials (every process forms the same norm, clip
 *      coefficient, scaler update and skip decision, bit for bit);
 *   5. zero_adamw_cast_gather_local on the local range;
 *   6. exchange: all-gather the local parameters into the full gathered buffer.
 * With the ranks' sums taken in ascending rank order in step 2 and the fixed-order sum of
 * step 4, every output equals the one-GPU step's (zero_step) bit for bit.
 * ------------------------------------------------------------------------------------- */

/* zero_reduce_shard_unscale on a window inside the local range, g stored locally.
 *   replicas   HOST array of N DEVICE pointers; replicas[k] points at flat element `begin`
 *              of rank k's gradient copy (e.g. inside the chunk received from rank k)
 *   begin      multiple of 8; [begin, begin + count) inside [origin, origin + local_len)
 *   g_local    DEVICE fp32, local_len elements: g of flat i is stored at g_local[i - origin]
 *   partials   DEVICE, zero_workspace_bytes(layout) (all ranks' slots); the local ranks'
 *              slots are accumulated as in zero_reduce_shard_unscale
 *   st         DEVICE step state of this process (its overflow word is set as there)
 * ZERO_EINVAL for a bad rank range or a window outside it. */
int zero_reduce_shard_unscale_local(const zero_layout_t* layout, zero_dtype_t dtype,
                                    uint32_t rank_begin, uint32_t rank_count,
                                    const void* const* replicas, uint64_t begin, uint64_t count,
                                    float* g_local, double* partials, zero_step_state_t* st,
                                    zero_stream_t stream);

/* zero_adamw_cast_gather on the local range only: element j of every local array is flat
 * origin + j; elements at flat >= psi are padding (parameters written 0, state untouched).
 *   g_local, master_local, m_local, v_local   DEVICE fp32, local_len elements each
 *   params_local   DEVICE 16-bit, local_len elements: this process's part of the gathered
 *                  buffer (it may point at flat `origin` of the full buffer, so that an
 *                  in-place all-gather completes it)
 *   st             DEVICE step state after zero_grad_norm of this step */
int zero_adamw_cast_gather_local(const zero_layout_t* layout, const zero_adamw_hparams_t* hp,
                                 uint32_t rank_begin, uint32_t rank_count, const float* g_local,
                                 float* master_local, float* m_local, float* v_local,
                                 uint16_t* params_local, const zero_step_state_t* st,
                                 zero_stream_t stream);

/* -------------------------------------------------------------------------------------
 * zero_step -- one whole step: every bucket's reduce, the norm, AdamW + cast.
 *   replicas   HOST array of n_buckets * N DEVICE pointers, bucket-major:
 *              replicas[b*N + k] holds rank k's gradient for flat
 *              [b*W, min((b+1)*W, psi_padded)).  With n_buckets = 1 these are simply
 *              the N full gradient copies.
 *   g          as in zero_reduce_shard_unscale, or NULL when N = 2 and n_buckets = 1:
 *              the re-reading schedule.  Clipping needs the global norm before any
 *              update, so an exact step either writes the fp32 g and reads it back
 *              (34 + 2N bytes per parameter) or reads the N copies twice (26 + 4N); at
 *              N = 2 the second moves 34 instead of 38 B.  The reduce then stores no g
 *              and AdamW forms each g[i] again from the two copies with the same
 *              arithmetic (same bits).  ZERO_EINVAL for NULL g with any other layout.
 *   other arguments as in the three calls above.
 * Launches: n_buckets + 2 kernels (the reduce per bucket, the norm, AdamW).  A small
 * layout (one bucket, at most 128 tile slots per rank, and every one of its n_tiles tiles
 * able to hold a resident block at once: up to a few million parameters) runs instead
 * as ONE cooperative kernel with the same bits: each block reduces one tile and keeps
 * its g in shared memory (with at most one tile per SM, also the tile's master, m and v,
 * bulk-copied in as the block starts), the block that finishes last forms the global norm
 * and the step's scalars, and every block then updates its tile.  g is still written when given
 * (never read back), so such a step moves 2N + 30 bytes per parameter, 2N + 26 with
 * g = NULL (+2 with at most one tile per SM: the gathered parameters are read too, so
 * that an update made ahead of the norm can be undone).  zero_step_launches tells which way a layout goes.  If the cooperative launch
 * is refused because fewer blocks fit on the GPU than its occupancy promised (another
 * context holds part of it), the same call makes the three launches instead.
 * ------------------------------------------------------------------------------------- */
int zero_step(const zero_layout_t* layout, const zero_adamw_hparams_t* hp, zero_dtype_t dtype,
              const void* const* replicas, float* g, double* partials, float* master, float* m,
              float* v, uint16_t* params, zero_step_state_t* st, zero_stream_t stream);

/* Kernel launches one zero_step call makes for this layout and gradient type on the
 * current device: 1 (the single-launch step) or n_buckets + 2.  ZERO_EINVAL (negative) for
 * an invalid layout or dtype.  Enqueues nothing; the first call on a device queries the
 * kernel's occupancy there. */
int zero_step_launches(const zero_layout_t* layout, zero_dtype_t dtype);

/* -------------------------------------------------------------------------------------
 * zero_step_host -- zero_step with the gradients in HOST memory.
 * The N gradient copies arrive from pinned host memory, one bucket of W elements at a
 * time, through a two-slot device staging ring: the copy of bucket b+1 (on copy_stream,
 * one cudaMemcpyAsync per rank) overlaps the reduce of bucket b (on stream).
 *   host_replicas   HOST array of N HOST pointers (pinned for overlap), each psi_padded
 *                   elements of dtype; read asynchronously, so they must stay unchanged
 *                   until the step has completed on `stream`
 *   staging         DEVICE buffer of staging_bytes >= 2 * N * W8 * sizeof(dtype), W8 = W
 *                   rounded up to a multiple of 8 (so every staged copy is 16-byte
 *                   aligned; W itself is a multiple of 8 whenever there are several
 *                   buckets); not touched when the copies are read in place
 *   host_state_out  optional HOST pointer (pinned): the step state is copied there at
 *                   the end of the step on `stream` (the caller synchronises)
 *   copy_stream     must differ from stream
 * A small layout in one bucket (one that zero_step runs as a single launch) runs as that
 * single launch here too.  When every copy lies in page-locked host memory (through its
 * whole psi_padded range, 16-byte aligned), the launch reads the copies there directly
 * over the CPU-GPU link, and staging is not touched; otherwise the copies are staged
 * first.
 * Returns ZERO_ENOMEM if staging is too small.
 * ------------------------------------------------------------------------------------- */
int zero_step_host(const zero_layout_t* layout, const zero_adamw_hparams_t* hp,
                   zero_dtype_t dtype, const void* const* host_replicas, void* staging,
                   uint64_t staging_bytes, float* g, double* partials, float* master, float* m,
                   float* v, uint16_t* params, zero_step_state_t* st,
                   zero_step_state_t* host_state_out, zero_stream_t stream,
                   zero_stream_t copy_stream);

/* -------------------------------------------------------------------------------------
 * zero_step_static_workspace -- zero_step for callers that cannot allocate device memory.
 * The ZeRO pages have no counterpart of this call; it exists for how the library is used.
 * Some callers cannot give the library a scratch buffer: their memory manager already
 * holds all of the GPU's memory, or they must not take the device-wide synchronisation
 * that a cudaMalloc or cudaFree can cause in the middle of a training step.  This call
 * runs the same step as zero_step, but keeps the step's only scratch, the per-tile
 * sum-of-squares partials, in a static device array of ZERO_STATIC_WORKSPACE_SLOTS
 * 8-byte slots (8 MiB) inside the library.  It calls no cudaMalloc, no cudaFree and no
 * other allocating routine.
 *   - The array is held on every GPU where the library's device code is loaded, from
 *     load until the process exits.
 *   - Layouts with n_tiles > ZERO_STATIC_WORKSPACE_SLOTS (more than about 8.6e9 padded
 *     parameters) are rejected with ZERO_ENOMEM before anything is enqueued.
 *   - The first call on each device looks up the array's device address (a one-time
 *     set-up, with that device current); make that first call before any stream capture
 *     begins.
 *   - Every call shares the one array and clears the slots it uses at its start, so two
 *     calls whose work overlaps on the GPU (different streams or threads) race: issue them
 *     one after another on one stream.
 *   - Arguments as in zero_step, without `partials`, except that g must not be NULL:
 *     this call has no re-reading schedule (ZERO_EINVAL for NULL g).  To initialise st
 *     with zero_step_state_init without allocating, pass any 16-byte-aligned device buffer
 *     of at least zero_workspace_bytes(layout) bytes as its `partials` argument, e.g. `g`
 *     whenever 4*psi_padded >= zero_workspace_bytes(layout), which holds for every shard
 *     size S >= 4 (every step overwrites g before reading it).
 *   - The address lookup is cached per device for the life of the process; after a
 *     cudaDeviceReset the library's device code may be loaded at another address, so do
 *     not call this entry point again in that process.
 * ------------------------------------------------------------------------------------- */
#define ZERO_STATIC_WORKSPACE_SLOTS (1u << 20)
int zero_step_static_workspace(const zero_layout_t* layout, const zero_adamw_hparams_t* hp,
                               zero_dtype_t dtype, const void* const* replicas, float* g,
                               float* master, float* m, float* v, uint16_t* params,
                               zero_step_state_t* st, zero_stream_t stream);

/* Text for a status code. */
const char* zero_strerror(int status);

/* cudaError_t of the last ZERO_ECUDA returned on this thread (0 if none). */
int zero_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_H */
