/*
 * reduce.cu -- reduce-scatter arithmetic, unscale, overflow flag, sum of squares.
 *
 * "【论文解读】ZeRO" sec. 6(1)-(2): data-parallel ranks average their gradients; with
 * gradient partitioning the average is reduce-scattered, so the owner of flat [r*S,(r+1)*S)
 * receives the mean of every rank's copy of that range (the page's 4-GPU example: GPU0
 * ends with G0,G1, GPU1 with G2,G3, ...).  All N ranks live on this GPU as N buffers, so
 * the collective's arithmetic is a streaming N-way sum:
 *
 *   g[i] = (x_0[i] + x_1[i] + ... + x_{N-1}[i]) * f32(1/(N*L))   (fp32, ascending rank)
 *
 * fused with the inf/NaN check of fp16 loss scaling and with the per-rank sum of g^2
 * that the global-norm all-reduce of the Megatron distributed-optimizer page (sec. 1)
 * combines.
 *
 * GB300 design.  Pure HBM streaming (2N bytes in, 4 out per element, a few flops), so:
 *  - a persistent grid (SM count x resident blocks) walks tiles of at most 8192
 *    elements: each shard cut at the flat multiples of 8192, so interior tiles start on
 *    128-byte lines of every array even when the shard size is not a multiple of 64
 *    (misaligned warps touched one extra line per load: 4% of the kernel's time at the
 *    GPT-2 size); one block owns a tile, so its partial gets exactly one add per launch
 *    (deterministic; the add is an fp64 atomicAdd only so that it need not wait);
 *  - every thread moves 8 elements per replica with one 128-bit non-coherent load that
 *    skips L1 (ld.global.nc.L1::no_allocate.v4), all N replica loads issued before the
 *    sum, and writes g with streaming 128-bit stores;
 *  - the sum of squares is carried per thread as two unevaluated fp32 pairs (even and odd
 *    elements) with error-free TwoProduct (FMA) and TwoSum steps, which keeps it at
 *    ~2^-48 relative accuracy without per-element fp64 (GB300's fp64 rate is a small
 *    fraction of fp32), then folded into fp64 once per warp and reduced in a fixed tree
 *    per tile; the rank sums, the unscale and both pairs' steps use Blackwell's paired
 *    fp32 instructions (two operations of one thread in one instruction, same bits);
 *  - groups with an element outside the pair arithmetic's exact range (below 2^-74 or
 *    at least 2^32 in magnitude, or not finite) are summed in fp64 instead;
 *  - launched with programmatic dependent launch (the kernel waits for the preceding grid
 *    first thing), so its launch overlaps the previous kernel's tail.
 */
#include "reduce_elem.cuh"

#include <atomic>

namespace zero {
namespace {

constexpr int kBlock = 256;
constexpr int kLoadBatch = 8;  // replica loads in flight per thread before summing
// with 8 copies the kernel is compiled for 5 resident blocks of 256 threads per SM (48
// registers; left to itself the compiler takes 56, which allows only 4); the other rank
// counts are left to the compiler (46-48 registers, 5 blocks; 74 and 3 for the generic
// kernel), where a bound made it spill
constexpr int kMinBlocksN8 = 5;

/* The tile j of rank r, clipped to the window: [lo, hi), empty for a rank's trailing
 * slot.  Shards are cut at the flat multiples of the tile size, so the 128-bit loads of
 * interior tiles start on 128-byte lines of every array. */
__device__ __forceinline__ void tile_bounds(const ReduceArgs& a, uint64_t unit, uint64_t& lo, uint64_t& hi)
{
    constexpr uint64_t T = ZERO_TILE_ELEMS;  // the layout's tile_elems (checked on the host)
    const uint64_t tpr = a.tiles_per_rank;
    // 64-bit division is a long instruction sequence; 32 bits cover any layout below
    // 2^32 tiles (3.5e13 parameters)
    const uint64_t r = (unit >> 32) == 0 && (tpr >> 32) == 0 ? (uint64_t)((uint32_t)unit / (uint32_t)tpr)
                                                              : unit / tpr;
    const uint64_t j = unit - r * tpr;
    const uint64_t shard_lo = r * a.shard, shard_hi = shard_lo + a.shard;
    const uint64_t cell = (shard_lo / T + j) * T;
    lo = cell > shard_lo ? cell : shard_lo;
    hi = cell + T < shard_hi ? cell + T : shard_hi;
    lo = lo > a.begin ? lo : a.begin;
    hi = hi < a.end ? hi : a.end;
}

/* Elements b .. b+7 once their rank sums s[] are known: the group's values, squares and
 * overflow check (group_values), then g stored. */
__device__ __forceinline__ void finish_group(const ReduceArgs& a, float inv, float (&s)[8], uint64_t b,
                                             uint64_t lo, uint64_t hi, SumSq& acc, bool& bad)
{
    float gv[8];
    uint32_t in;
    bool full;
    group_values(a.psi, inv, s, b, lo, hi, acc, bad, gv, in, full);
    if (!a.g) {
        // no g: the AdamW pass re-reads the gradient copies instead (small N)
    } else if (full) {
        if (ZERO_OWNED(b, 8, lo, hi, &a.st->error)) {
            __stcs(reinterpret_cast<float4*>(a.g + b), make_float4(gv[0], gv[1], gv[2], gv[3]));
            __stcs(reinterpret_cast<float4*>(a.g + b + 4), make_float4(gv[4], gv[5], gv[6], gv[7]));
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if ((in >> e & 1u) && ZERO_OWNED(b + e, 1, lo, hi, &a.st->error))
                a.g[b + e] = gv[e];
    }
}

/* One tile straight from the replicas: 8 elements per 128-bit load per replica, all N
 * loads of a group issued before the ordered sum. */
template <zero_dtype_t DT, int NR>
__device__ __forceinline__ void tile_ldg(const ReduceArgs& a, float inv, uint64_t lo, uint64_t hi,
                                         SumSq& acc, bool& bad)
{
    const int N = NR > 0 ? NR : (int)a.n_ranks;
    for (uint64_t b = (lo & ~7ull) + 8ull * threadIdx.x; b < hi; b += 8ull * kBlock) {
        float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const uint64_t off = b - a.begin;  // a multiple of 8: begin is
        if (b + 8 <= a.end) {
            // the whole group lies inside the window's buffers: 128-bit loads, even where it
            // straddles a tile edge (the other tile's elements are masked)
#pragma unroll 1
            for (int k0 = 0; k0 < N; k0 += kLoadBatch) {
                uint4 v[kLoadBatch];
#pragma unroll
                for (int kk = 0; kk < kLoadBatch; ++kk)
                    if (NR > 0 ? (k0 + kk < NR) : (k0 + kk < N))
                        v[kk] = ld_stream_v4((const uint16_t*)a.rep[k0 + kk] + off);
#pragma unroll
                for (int kk = 0; kk < kLoadBatch; ++kk)
                    if (NR > 0 ? (k0 + kk < NR) : (k0 + kk < N))
                        add8<DT>(s, v[kk]);
            }
        } else {  // the window's last, ragged group: element loads inside [lo, hi) only
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint64_t i = b + e;
                if (i >= lo && i < hi)
                    for (int k = 0; k < N; ++k)
                        s[e] = __fadd_rn(s[e], one16<DT>(ld_stream_u16((const uint16_t*)a.rep[k] + off + e)));
            }
        }
        finish_group(a, inv, s, b, lo, hi, acc, bad);
    }
}

/* The tile's partial (tile_fold: a fixed-order tree, fp64 once per warp, the warps in
 * order), added to the tile's slot.  The add is an fp64 atomicAdd whose result is not
 * used, so thread 0 does not wait for the old value.  Only one block adds to a tile in a
 * launch, and the windows of a step meet a tile in stream order, so the sum's order, and
 * its bits, are fixed. */
__device__ __forceinline__ void tile_done(const ReduceArgs& a, uint64_t unit, const SumSq& acc,
                                          WarpPart (*warp_part)[kBlock / 32], uint32_t& parity)
{
    const double t = tile_fold<kBlock>(acc, warp_part, parity);
    if (threadIdx.x == 0)
        atomicAdd(a.partials + unit, t);
}

/* The reduce: a persistent grid over the window's tiles, one block per tile at a time. */
template <zero_dtype_t DT, int NR>
__global__ void __launch_bounds__(kBlock, NR == 8 ? kMinBlocksN8 : 0 /* unbounded */) k_reduce(const __grid_constant__ ReduceArgs a)
{
    grid_dependency_wait();
    const float inv = a.st->inv_scale;
    __shared__ WarpPart warp_part[2][kBlock / 32];
    uint32_t parity = 0;
    bool bad = false;
    for (uint64_t u = blockIdx.x; u < a.unit_count; u += gridDim.x) {
        const uint64_t unit = a.unit_first + u;
        uint64_t lo, hi;
        tile_bounds(a, unit, lo, hi);
        if (lo >= hi)  // a rank's trailing empty slot, or a tile outside the window
            continue;
        SumSq acc;
        tile_ldg<DT, NR>(a, inv, lo, hi, acc, bad);
        tile_done(a, unit, acc, warp_part, parity);
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0)
        atomicOr(&a.st->overflow, 1u);
}

template <zero_dtype_t DT, int NR>
cudaError_t launch_t(const ReduceArgs& a, cudaStream_t s)
{
    static std::atomic<int> per_sm[64];  // per device; a race only repeats the query
    int dev = 0;
    cudaGetDevice(&dev);
    int occ = per_sm[dev & 63].load(std::memory_order_relaxed);
    if (occ == 0) {
        int o = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, k_reduce<DT, NR>, kBlock, 0);
        occ = o > 0 ? o : 1;
        per_sm[dev & 63].store(occ, std::memory_order_relaxed);
    }
    const uint64_t cap = (uint64_t)sm_count() * (uint64_t)occ;
    const unsigned grid = (unsigned)(a.unit_count < cap ? a.unit_count : cap);
    if (grid == 0)
        return cudaSuccess;
    return launch_pdl(k_reduce<DT, NR>, dim3(grid), dim3(kBlock), 0, s, a);
}

template <zero_dtype_t DT>
cudaError_t launch_dt(const ReduceArgs& a, cudaStream_t s)
{
    switch (a.n_ranks) {
    case 2: return launch_t<DT, 2>(a, s);
    case 4: return launch_t<DT, 4>(a, s);
    case 8: return launch_t<DT, 8>(a, s);
    case 16: return launch_t<DT, 16>(a, s);
    default: return launch_t<DT, 0>(a, s);
    }
}

#ifdef ZERO_TEST_HOOKS
/* Test builds only (never the product library): the exact-range test of the sum of
 * squares on n groups of 8 values, one thread per group, so that a test can compare the
 * device's decisions with the test's integer definition. */
__global__ void k_test_squares_in_range(const float* x, uint8_t* out, uint64_t n)
{
    const uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n)
        return;
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        v[e] = x[8 * i + e];
    out[i] = squares_in_range(v) ? 1 : 0;
}
#endif

}  // namespace

#ifdef ZERO_TEST_HOOKS
extern "C" int zero_test_squares_in_range(const float* x, uint8_t* out, unsigned long long n)
{
    if (n == 0)
        return 0;
    k_test_squares_in_range<<<(unsigned)((n + 255) / 256), 256>>>(x, out, n);
    return cudaGetLastError() == cudaSuccess && cudaDeviceSynchronize() == cudaSuccess ? 0 : -4;
}
#endif

cudaError_t launch_reduce(const ReduceArgs& a, zero_dtype_t dtype, cudaStream_t s)
{
    return dtype == ZERO_F16 ? launch_dt<ZERO_F16>(a, s) : launch_dt<ZERO_BF16>(a, s);
}

}  // namespace zero
