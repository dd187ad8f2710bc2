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
 *  - the sum of squares is carried per thread as an unevaluated fp32 pair with error-free
 *    TwoProduct (FMA) and TwoSum steps, which keeps it at ~2^-48 relative accuracy without
 *    per-element fp64 (GB300's fp64 rate is a small fraction of fp32), then folded into
 *    fp64 once per thread and reduced in a fixed shuffle tree per tile;
 *  - groups with an element outside the pair arithmetic's exact range (below 2^-74 or
 *    at least 2^34 in magnitude, or not finite) are summed in fp64 instead;
 *  - launched with programmatic dependent launch (the kernel waits for the preceding grid
 *    first thing), so its launch overlaps the previous kernel's tail.
 */
#include "zero_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace zero {
namespace {

constexpr int kBlock = 256;
constexpr int kLoadBatch = 8;  // replica loads in flight per thread before summing

template <zero_dtype_t DT>
__device__ __forceinline__ float lo16(uint32_t w);
template <zero_dtype_t DT>
__device__ __forceinline__ float hi16(uint32_t w);

template <>
__device__ __forceinline__ float lo16<ZERO_BF16>(uint32_t w) { return __uint_as_float(w << 16); }
template <>
__device__ __forceinline__ float hi16<ZERO_BF16>(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
template <>
__device__ __forceinline__ float lo16<ZERO_F16>(uint32_t w)
{
    return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
}
template <>
__device__ __forceinline__ float hi16<ZERO_F16>(uint32_t w)
{
    return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}

template <zero_dtype_t DT>
__device__ __forceinline__ float one16(uint16_t b)
{
    return lo16<DT>((uint32_t)b);
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ uint16_t ld_stream_u16(const void* p)
{
    unsigned short v;
    asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

template <zero_dtype_t DT>
__device__ __forceinline__ void add8(float (&s)[8], const uint4& v)
{
    s[0] = __fadd_rn(s[0], lo16<DT>(v.x));
    s[1] = __fadd_rn(s[1], hi16<DT>(v.x));
    s[2] = __fadd_rn(s[2], lo16<DT>(v.y));
    s[3] = __fadd_rn(s[3], hi16<DT>(v.y));
    s[4] = __fadd_rn(s[4], lo16<DT>(v.z));
    s[5] = __fadd_rn(s[5], hi16<DT>(v.z));
    s[6] = __fadd_rn(s[6], lo16<DT>(v.w));
    s[7] = __fadd_rn(s[7], hi16<DT>(v.w));
}

/* Sum of squares of the fp32 gradient, carried as an unevaluated pair hi + lo of fp32
 * values.  TwoProduct: x*x = p + pe exactly (FMA); TwoSum: hi + p = s + err exactly.
 * The values are scaled by 2^24 first (exact) and the tile's total by 2^-48 at the end,
 * which moves the range where every step is exact and nothing can overflow (1024 squares
 * per warp before the fp64 fold) to |x| in [2^-74, 2^34), plus zeros: gradients of
 * ~1e-4 often come within 2^-50 of zero, which unscaled would need the fp64 path.
 * Power-of-two scaling changes no rounding, so the result is the unscaled pair sum's.
 * Groups holding anything outside that range take the fp64 path below. */
constexpr float kSqScale = 16777216.0f;  // 2^24
constexpr double kSqUnscale = 0x1p-48;
struct SumSq {
    float hi = 0.0f, lo = 0.0f;
    double wide = 0.0;

    __device__ __forceinline__ void add_fast(float x)
    {
        const float p = __fmul_rn(x, x);
        const float pe = __fmaf_rn(x, x, -p);
        const float s = __fadd_rn(hi, p);
        const float bb = __fsub_rn(s, hi);
        const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(p, bb));
        hi = s;
        lo = __fadd_rn(lo, __fadd_rn(err, pe));
    }
};

/* True when all 8 values are finite and every scaled square is exact in the fp32 pair
 * arithmetic: magnitudes in [2^-74, 2^34) or zero.  Integer compares on the magnitude
 * bits, so NaN (above inf) and inf fail the test too. */
__device__ __forceinline__ bool squares_in_range(const float (&x)[8])
{
    uint32_t mx = 0u, mn = 0x3f800000u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t u = __float_as_uint(x[e]) & 0x7fffffffu;
        mx = max(mx, u);
        mn = min(mn, u == 0u ? 0x3f800000u : u);
    }
    return mx < 0x50800000u && mn >= 0x1a800000u;  // 2^34 and 2^-74
}

/* fp64 sum of squares of the elements of a group selected by mask; a real call, so the
 * fp64 work runs only for the rare groups that need it. */
__device__ __noinline__ double sumsq_wide(float x0, float x1, float x2, float x3, float x4, float x5,
                                          float x6, float x7, uint32_t mask)
{
    const float x[8] = {x0, x1, x2, x3, x4, x5, x6, x7};
    double t = 0.0;
    for (int e = 0; e < 8; ++e)
        if (mask >> e & 1u)
            t += (double)x[e] * (double)x[e];
    return t;
}

/* hi1 + lo1 += hi2 + lo2 in pair arithmetic (TwoSum on the leading parts). */
__device__ __forceinline__ void pair_add(float& hi, float& lo, float h2, float l2)
{
    const float s = __fadd_rn(hi, h2);
    const float bb = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(h2, bb));
    hi = s;
    lo = __fadd_rn(__fadd_rn(lo, l2), err);
}

__device__ __forceinline__ bool not_finite(float x)
{
    return (__float_as_uint(x) & 0x7f800000u) == 0x7f800000u;
}

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

/* Elements b .. b+7 once their rank sums s[] are known: unscale, zero the padding, mask
 * what lies outside the tile [lo, hi), add the squares, flag non-finite values, store g. */
__device__ __forceinline__ void finish_group(const ReduceArgs& a, float inv, float (&s)[8], uint64_t b,
                                             uint64_t lo, uint64_t hi, SumSq& acc, bool& bad)
{
    const bool full = b >= lo && b + 8 <= hi;  // all 8 elements belong to this tile
    float gv[8], sq[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        gv[e] = sq[e] = __fmul_rn(s[e], inv);
    uint32_t in = 0xffu;
    if (b + 8 > a.psi || !full) {  // padding, or a group cut by the tile/window edge
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint64_t i = b + e;
            if (i >= a.psi)
                gv[e] = 0.0f;
            if (!(i >= lo && i < hi))
                in &= ~(1u << e);
            sq[e] = (in >> e & 1u) ? gv[e] : 0.0f;
        }
    }
    if (squares_in_range(sq)) {  // every counted element finite: no overflow
#pragma unroll
        for (int e = 0; e < 8; ++e)
            acc.add_fast(__fmul_rn(sq[e], kSqScale));
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            bad |= (in >> e & 1u) && not_finite(gv[e]);
        acc.wide += sumsq_wide(gv[0], gv[1], gv[2], gv[3], gv[4], gv[5], gv[6], gv[7], in);
    }
    if (!a.g) {
        // no g: the AdamW pass re-reads the gradient copies instead (small N)
    } else if (full) {
        __stcs(reinterpret_cast<float4*>(a.g + b), make_float4(gv[0], gv[1], gv[2], gv[3]));
        __stcs(reinterpret_cast<float4*>(a.g + b + 4), make_float4(gv[4], gv[5], gv[6], gv[7]));
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (in >> e & 1u)
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

/* The tile's partial: a fixed-order pair-arithmetic shuffle tree in fp32, fp64 once per
 * warp, the warps in order, added to the tile's slot.  One block barrier; the per-warp
 * values alternate between two buffers (tile parity), so the next tile cannot overwrite
 * them before thread 0 has read them.  The add is an fp64 atomicAdd whose result is not
 * used, so thread 0 does not wait for the old value.  Only one block adds to a tile in a
 * launch, and the windows of a step meet a tile in stream order, so the sum's order, and
 * its bits, are fixed. */
__device__ __forceinline__ void tile_done(const ReduceArgs& a, uint64_t unit, const SumSq& acc,
                                          double (*warp_part)[kBlock / 32], uint32_t& parity)
{
    float ph = acc.hi, pl = acc.lo;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float h2 = __shfl_xor_sync(0xffffffffu, ph, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, pl, o);
        pair_add(ph, pl, h2, l2);
    }
    double wide = acc.wide;
    if (__any_sync(0xffffffffu, wide != 0.0)) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            wide += __shfl_xor_sync(0xffffffffu, wide, o);
    }
    double* wp = warp_part[parity];
    if ((threadIdx.x & 31) == 0)
        wp[threadIdx.x >> 5] = ((double)ph + (double)pl) * kSqUnscale + wide;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
#pragma unroll
        for (int w = 0; w < kBlock / 32; ++w)
            t += wp[w];
        atomicAdd(a.partials + unit, t);
    }
    parity ^= 1u;
}

/* The reduce: a persistent grid over the window's tiles, one block per tile at a time. */
template <zero_dtype_t DT, int NR>
__global__ void __launch_bounds__(kBlock) k_reduce(const __grid_constant__ ReduceArgs a)
{
    grid_dependency_wait();
    const float inv = a.st->inv_scale;
    __shared__ double warp_part[2][kBlock / 32];
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
    static int per_sm[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int& occ = per_sm[dev & 63];
    if (occ == 0) {
        int o = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, k_reduce<DT, NR>, kBlock, 0);
        occ = o > 0 ? o : 1;
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

}  // namespace

cudaError_t launch_reduce(const ReduceArgs& a, zero_dtype_t dtype, cudaStream_t s)
{
    return dtype == ZERO_F16 ? launch_dt<ZERO_F16>(a, s) : launch_dt<ZERO_BF16>(a, s);
}

}  // namespace zero
