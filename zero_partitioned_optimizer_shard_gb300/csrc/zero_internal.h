/*
 * zero_internal.h -- shared declarations of the CUDA library behind include/zero.h.
 */
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/zero.h"

namespace zero {

/* Kernel arguments of the reduce-scatter / unscale / sum-of-squares pass. */
struct ReduceArgs {
    const void* rep[ZERO_MAX_KERNEL_RANKS];  // replica k, pointing at flat `begin`
    float* g;                                // flat fp32 gradient, psi_padded
    double* partials;                        // one fp64 slot per tile (shards cut on the flat T grid)
    zero_step_state_t* st;
    uint64_t begin, end;                     // window [begin, end)
    uint64_t psi, shard;
    uint64_t tiles_per_rank;
    uint64_t unit_first, unit_count;         // tile slots that meet the window
    uint32_t n_ranks;
    uint32_t tile;
};

struct FinalizeArgs {
    double* partials;
    zero_step_state_t* st;
    uint64_t tiles_per_rank;
    uint32_t n_ranks;
    zero_adamw_hparams_t hp;
};

struct AdamwArgs {
    const float* g;
    float* master;
    float* m;
    float* v;
    uint16_t* out;
    const zero_step_state_t* st;
    uint32_t* err;                           // the state's error word (bounded waits)
    unsigned long long* next_chunk;          // the state's adamw_next_chunk (k_adamw's queue)
    uint32_t* done;                          // the state's adamw_done
    uint64_t psi, psi_padded;
    float beta1, beta2, eps;
    uint32_t out_f16;                        // gathered parameters as fp16 instead of bf16
    // re-reading schedule (N = 2, g not materialised): the two gradient copies instead of g
    const uint16_t* rep0;
    const uint16_t* rep1;
    uint32_t grad_f16;                       // copies are fp16 (else bf16)
};

static_assert(sizeof(zero_step_state_t) == 128, "the step state is 128 bytes");
static_assert(offsetof(zero_step_state_t, adamw_next_chunk) % 8 == 0, "the chunk queue is 8-byte aligned");
// the single launch's arrival counter and the step's outcome form one 64-bit word
// (counter in the low half), written at once when the last block releases the others
static_assert(offsetof(zero_step_state_t, launch_arrivals) % 8 == 0 &&
                  offsetof(zero_step_state_t, applied_c) == offsetof(zero_step_state_t, launch_arrivals) + 4,
              "launch_arrivals and applied_c share one aligned 64-bit word");

/* Kernel arguments of the single-launch step for small layouts (fused.cu). */
struct FusedArgs {
    const void* rep[ZERO_MAX_KERNEL_RANKS];  // replica k, pointing at flat 0
    float* g;                                // flat fp32 gradient, or null: not written
    double* partials;                        // the tile partials: zero on entry and on exit
    float* master;
    float* m;
    float* v;
    uint16_t* out;
    zero_step_state_t* st;
    uint64_t psi, psi_padded, shard, tiles_per_rank;
    uint32_t n_ranks;
    uint32_t out_f16;                        // gathered parameters as fp16 instead of bf16
    zero_adamw_hparams_t hp;
};

/* The single-launch step takes layouts of at most this many tile slots per rank (the norm
 * kernel then sums each rank's slots in one lane-strided pass) whose n_tiles blocks can
 * all be resident at once. */
constexpr uint64_t kFusedMaxTilesPerRank = 128;

struct InitArgs {
    zero_step_state_t* st;
    double* partials;
    uint64_t n_tiles;
    float loss_scale;
    uint32_t dynamic, growth_interval, n_ranks;
};

/* Programmatic dependent launch (Hopper/Blackwell): the kernel may be launched while the
 * preceding kernel in the stream is still finishing, so the launch itself overlaps that
 * kernel's tail.  Every kernel launched this way executes grid_dependency_wait() as its
 * first instruction, which returns once the preceding grid has completed and its memory
 * is visible: nothing runs early, so stream order holds whatever the preceding kernel is. */
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

/* Lets the next kernel in the stream (launched with programmatic dependent launch) start
 * now: its blocks become resident and wait in grid_dependency_wait() until this grid has
 * completed, so no launch latency is left between the two. */
__device__ __forceinline__ void grid_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

/* An NVTX range named after an entry point, over its host-side work (checks and launches),
 * so profilers can attribute and filter its kernels (e.g. ncu --nvtx --nvtx-include
 * "zero_step/").  NVTX v3 is header-only: with no tool attached a range costs a few
 * nanoseconds and loads nothing. */
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

/* Checked builds (-DZERO_CHECKED, made by a test; never the product library): before each
 * store of the reduce pass and of the single-launch step, ZERO_OWNED checks that elements
 * [i, i+n) lie in [lo, hi), the range the storing block owns; a failed check records 2 in
 * the step state's error word and the store is skipped, so an indexing mistake shows up
 * as a status, not as a fault or a silently overwritten neighbour.  In the product build
 * the check is the constant true and costs nothing. */
#ifdef ZERO_CHECKED
__device__ __forceinline__ bool zero_owned(uint64_t i, uint64_t n, uint64_t lo, uint64_t hi,
                                           uint32_t* err)
{
    if (i >= lo && i + n <= hi)
        return true;
    atomicOr(err, 2u);
    return false;
}
#define ZERO_OWNED(i, n, lo, hi, err) zero_owned((i), (n), (lo), (hi), (err))
#else
#define ZERO_OWNED(i, n, lo, hi, err) true
#endif

/* Launchers (enqueue only; return the launch's cudaError_t). */
cudaError_t launch_reduce(const ReduceArgs& a, zero_dtype_t dtype, cudaStream_t s);
cudaError_t launch_finalize(const FinalizeArgs& a, cudaStream_t s);
cudaError_t launch_adamw(const AdamwArgs& a, cudaStream_t s);
cudaError_t launch_adamw_host_state(const AdamwArgs& a, cudaStream_t s);
cudaError_t launch_adamw_rereduce(const AdamwArgs& a, cudaStream_t s);  // g from rep0 + rep1  // master/m/v in pinned host memory
cudaError_t launch_state_init(const InitArgs& a, cudaStream_t s);
/* Which single-launch shape a layout takes: 0 none (the three-launch step), 1 unstaged
 * (up to 3 blocks per SM), 2 staged (one block per SM, the tile's optimizer state in
 * shared memory). */
int fused_shape(const zero_layout_t* L, zero_dtype_t dtype);
cudaError_t launch_step_fused(const FusedArgs& a, zero_dtype_t dtype, uint64_t n_tiles, int shape,
                              cudaStream_t s);

/* Resident blocks per SM times SM count for a kernel, cached per device. */
bool layout_ok(const zero_layout_t* L);  // the invariants zero_partition establishes

/* Sum-of-squares tiles: each shard [r*S, (r+1)*S) cut at the flat multiples of T, so
 * every interior tile starts on a 128-byte line of each array whatever S is.  Tile j of
 * rank r = [r*S, (r+1)*S) intersected with [(c+j)*T, (c+j+1)*T), c = floor(r*S/T);
 * partial slot r*tiles_per_rank + j (trailing slots of a rank may be empty). */
uint64_t tiles_per_rank(uint64_t S, uint64_t T);
uint64_t tile_unit(const zero_layout_t* L, uint64_t i);  // slot of the tile holding flat i
int sm_count();

/* Whether an AdamW pass moving bytes_per_elem bytes for each of n elements should bulk-load
 * under an L2 evict-first policy: when its data is at least 16 times the L2 of the current
 * device.  Measured on GB300 (126 MB of L2): from 2^26 parameters up the policy is as fast
 * or faster (2^28: 2.4%, the GPT-2-1.5B buffer: 4%); at 2^22-2^25 it cost 1-3%. */
bool adamw_evict_first(uint64_t n, uint64_t bytes_per_elem);

/* Make zero_last_cuda_error() report `e` on this thread. */
void record_cuda_error(int e);

}  // namespace zero
