/*
 * finalize.cu -- global gradient norm, clip coefficient, loss scaler, skip decision.
 *
 * The Megatron distributed-optimizer page (gitcode.csdn.net, sec. 1, AdamW global
 * grad_norm table): inside optimizer.step(), before gradients are clipped, one all-reduce
 * turns the ranks' local squared norms into the global L2 norm that sets clip_coeff.  With
 * the ranks on one GPU that all-reduce is a fixed-order sum: each rank's tile partials
 * (written by the reduce pass) are summed per rank, then the ranks in order.
 *
 * The scaler follows fp16 mixed-precision training ("3、ZeRO技术概述" DeepSpeed config,
 * "fp16": enabled): a step whose reduced gradient holds inf/NaN is skipped and a dynamic
 * loss scale halves (floor 1); every growth_interval consecutive good steps it doubles
 * (cap 2^24).  Everything stays on the device, so a training loop never waits for the
 * host between steps.
 *
 * One extra block runs everything that does not need the norm (skip, t, the scaler, the
 * bias corrections with their two fp64 powers of beta, which GB300's slow fp64 pipe
 * makes the longest chain), split over three warps, beside the sums.  The last block to arrive
 * then only takes the square root and the clip coefficient.
 *
 * The sum is spread over up to 128 blocks, one warp per rank in each: block b sums the
 * fixed chunk b of every rank's tile partials (each lane in order, then a fixed shuffle
 * tree), leaves that chunk's sum in the chunk's first slot and zeroes the rest; the last
 * block to arrive (an atomic counter in the step state, no waiting) adds the chunk sums
 * of each rank in order, then the ranks in order.  GB300's fp64 rate is a few
 * operations per SM per clock, so the work is shaped to need few of them: one
 * accumulator per warp (eight per warp measured 7 us at a million parameters, against
 * about 1.5 us now).  The chunking depends only on N and the tile count, so the result
 * is the same on any GPU.  All partial slots end at zero, ready for the next step's
 * reduce windows.
 */
#include "step_scalars.cuh"

namespace zero {
namespace {

constexpr int kFinThreads = 256;
constexpr int kFinWarps = kFinThreads / 32;
constexpr int kFinMaxBlocks = 128;  // summing blocks; one more block runs the scalar logic

__global__ void __launch_bounds__(kFinThreads) k_finalize(const __grid_constant__ FinalizeArgs a)
{
    __shared__ double rank_sum[ZERO_MAX_KERNEL_RANKS];
    __shared__ int is_last;
    grid_dependency_wait();
    const uint32_t N = a.n_ranks;
    const uint64_t tpr = a.tiles_per_rank;
    const unsigned n_sum = gridDim.x - 1;  // blocks 0 .. n_sum-1 sum; block n_sum: scalars
    const uint64_t chunk = (tpr + n_sum - 1) / n_sum;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    zero_step_state_t* st = a.st;

    if (blockIdx.x == n_sum) {
        // Everything that does not need the norm, in three warps at once, beside the sums
        // (the two fp64 powers of beta are the longest chain on the slow fp64 pipe).  It
        // depends only on t and on the overflow flag, which every reduce window has set.
        __shared__ uint32_t s_t, s_overflow;
        if (threadIdx.x == 0) {
            s_t = st->t;
            s_overflow = st->overflow != 0;
        }
        __syncthreads();
        const uint32_t t = s_t + 1;  // the step count if this step is applied
        if (lane == 0 && w == 1 && !s_overflow)
            st->step_size = bias_step_size(a.hp, t);
        if (lane == 0 && w == 2 && !s_overflow)
            st->rbc2 = bias_rbc2(a.hp, t);
        if (lane == 0 && w == 3)
            scaler_update(st, a.hp, N, s_overflow, t);
    } else {
        // this block's chunk [j0, j1) of every rank's tile partials: one warp per rank,
        // each lane adds its slots in order, a fixed shuffle tree folds the warp.  The
        // chunk's sum is left in its first slot; the other slots are zeroed.
        const uint64_t j0 = (uint64_t)blockIdx.x * chunk;
        const uint64_t j1 = j0 + chunk < tpr ? j0 + chunk : tpr;
        for (uint32_t r = w; r < N; r += kFinWarps) {
            double* p = a.partials + (uint64_t)r * tpr;
            double acc = 0.0;
            for (uint64_t j = j0 + lane; j < j1; j += 32) {
                acc += p[j];
                p[j] = 0.0;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0 && j0 < j1)
                p[j0] = acc;
        }
    }
    // arrival: the block's writes are ordered before the count by the barrier and one
    // release fence of thread 0 (fences in every thread stalled the kernel on membar);
    // the last block to arrive acquires before reading the other blocks' chunk sums
    __syncthreads();
    if (threadIdx.x == 0) {
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        is_last = atomicAdd(&a.st->arrivals, 1u) == gridDim.x - 1;
        if (is_last)
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
    }
    __syncthreads();
    if (!is_last)
        return;

    // the last block: chunk sums in order per rank (one warp per rank), ranks in order
    const uint64_t n_chunks = (tpr + chunk - 1) / chunk;  // at most kFinMaxBlocks = 4 x 32
    for (uint32_t r = w; r < N; r += kFinWarps) {
        double* p = a.partials + (uint64_t)r * tpr;
        double v[kFinMaxBlocks / 32];
#pragma unroll
        for (int q = 0; q < kFinMaxBlocks / 32; ++q) {
            const uint64_t c = lane + 32u * q;
            v[q] = c < n_chunks ? __ldcg(p + c * chunk) : 0.0;
        }
        double s = 0.0;
#pragma unroll
        for (int q = 0; q < kFinMaxBlocks / 32; ++q) {
            const uint64_t c = lane + 32u * q;
            if (c < n_chunks) {
                s += v[q];
                p[c * chunk] = 0.0;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0)
            rank_sum[r] = s;
    }
    __syncthreads();
    if (threadIdx.x != 0)
        return;
    double total = 0.0;
    for (uint32_t r = 0; r < N; ++r)
        total += rank_sum[r];

    // the skip decision and the rest were written by the scalar block before it arrived
    st->arrivals = 0;
    const double norm = sqrt(total);
    st->sumsq = total;
    st->norm = norm;
    const uint32_t skip = __ldcg(&st->skip);
    const float c = clip_coefficient(norm, skip, a.hp.max_grad_norm);
    st->clip_coef = c;
    st->applied_c = skip ? -1.0f : c;
    st->overflow = 0;
    st->n_steps += 1;
}

__global__ void k_state_init(const __grid_constant__ InitArgs a)
{
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.n_tiles; i += stride)
        a.partials[i] = 0.0;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        zero_step_state_t s;
        memset(&s, 0, sizeof s);
        s.clip_coef = 1.0f;
        s.loss_scale = a.loss_scale;
        s.inv_scale = (float)(1.0 / ((double)a.n_ranks * (double)a.loss_scale));
        s.rbc2 = 1.0f;
        s.decay = 1.0f;
        s.dynamic = a.dynamic;
        s.growth_interval = a.growth_interval;
        s.n_ranks = a.n_ranks;
        *a.st = s;
    }
}

}  // namespace

cudaError_t launch_finalize(const FinalizeArgs& a, cudaStream_t s)
{
    uint64_t blocks = a.tiles_per_rank < (uint64_t)kFinMaxBlocks ? a.tiles_per_rank
                                                                 : (uint64_t)kFinMaxBlocks;
    if (blocks == 0)
        blocks = 1;
    return launch_pdl(k_finalize, dim3((unsigned)blocks + 1), dim3(kFinThreads), 0, s, a);
}

cudaError_t launch_state_init(const InitArgs& a, cudaStream_t s)
{
    const uint64_t want = (a.n_tiles + 255) / 256;
    const uint64_t cap = (uint64_t)sm_count() * 4;
    unsigned grid = (unsigned)(want < cap ? want : cap);
    if (grid == 0)
        grid = 1;
    k_state_init<<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace zero
