/*
 * reduce_elem.cuh -- the element arithmetic of the reduce-scatter pass, shared by the
 * reduce kernel (reduce.cu) and the single-launch step for small layouts (fused.cu), so
 * both compute the same bits: 16-bit gradient decoding, streaming loads, the rank-ordered
 * fp32 sum, the unscaled group values with their padding and tile masks, the error-free
 * sum of squares and its fixed-order fold per tile.
 */
#pragma once

#include "zero_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace zero {
namespace {

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

/* Two fp32 values in one 64-bit register, and Blackwell's paired fp32 arithmetic on them
 * (add/sub/mul .rn.f32x2): each half is the correctly rounded result of the scalar
 * operation, so a pair of scalar computations done this way keeps its bits, in half the
 * instructions. */
__device__ __forceinline__ uint64_t f2(float a, float b)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_split(uint64_t r, float& a, float& b)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

/* s[e] += x[e] for the 8 values of one 128-bit load of a copy, in fp32 pairs. */
template <zero_dtype_t DT>
__device__ __forceinline__ void add8(float (&s)[8], const uint4& v)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
        f2_split(f2_add(f2(s[2 * q], s[2 * q + 1]), f2(lo16<DT>(w[q]), hi16<DT>(w[q]))),
                 s[2 * q], s[2 * q + 1]);
}

/* Sum of squares of the fp32 gradient, carried as an unevaluated pair hi + lo of fp32
 * values.  TwoProduct: x*x = p + pe exactly (FMA); TwoSum: hi + p = s + err exactly.
 * The values are scaled by 2^24 first (exact) and the tile's total by 2^-48 at the end,
 * which moves the range where every step is exact and nothing can overflow (8192 squares
 * per tile before the fp64 conversion) to |x| in [2^-74, 2^32), plus zeros: gradients of
 * ~1e-4 often come within 2^-50 of zero, which unscaled would need the fp64 path.
 * Power-of-two scaling changes no rounding, so the result is the unscaled pair sum's.
 * Groups holding anything outside that range take the fp64 path below. */
constexpr float kSqScale = 16777216.0f;  // 2^24
constexpr double kSqUnscale = 0x1p-48;
/* Two such pairs per thread, one for the even and one for the odd elements of its groups,
 * each updated with the scalar steps, side by side in fp32x2 arithmetic (hi2, lo2 hold
 * the even pair's parts in their low halves, the odd pair's in their high halves);
 * tile_fold adds the two pairs first. */
struct SumSq {
    uint64_t hi2 = 0, lo2 = 0;  // +0.0f in both halves
    double wide = 0.0;

    /* x2: two scaled values, (even, odd).  The products' rounding errors x*x - p are
     * formed with scalar FMAs (as many instructions as the paired negation and FMA): a
     * paired FMA whose addend was a paired 0 - p gave wrong errors on GB300 in this
     * kernel, while every paired operation here matched its scalar twin on its own. */
    __device__ __forceinline__ void add_pair(uint64_t x2)
    {
        const uint64_t p = f2_mul(x2, x2);
        float x0, x1, p0, p1;
        f2_split(x2, x0, x1);
        f2_split(p, p0, p1);
        const uint64_t pe = f2(__fmaf_rn(x0, x0, -p0), __fmaf_rn(x1, x1, -p1));  // exact
        const uint64_t s = f2_add(hi2, p);
        const uint64_t bb = f2_sub(s, hi2);
        const uint64_t err = f2_add(f2_sub(hi2, f2_sub(s, bb)), f2_sub(p, bb));
        hi2 = s;
        lo2 = f2_add(lo2, f2_add(err, pe));
    }
};

/* True when all 8 values are finite and every scaled square is exact in the fp32 pair
 * arithmetic: magnitudes in [2^-74, 2^32) or zero.  Integer compares on the magnitude
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
    return mx < 0x4f800000u && mn >= 0x1a800000u;  // 2^32 and 2^-74
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

/* Elements b .. b+7 once their rank sums s[] are known: unscale (gv), zero the padding,
 * mask what lies outside the tile [lo, hi) (bit e of `in` set for the tile's elements),
 * add the tile's squares to acc and flag its non-finite values.  `full`: all 8 elements
 * belong to the tile. */
__device__ __forceinline__ void group_values(uint64_t psi, float inv, const float (&s)[8], uint64_t b,
                                             uint64_t lo, uint64_t hi, SumSq& acc, bool& bad,
                                             float (&gv)[8], uint32_t& in, bool& full)
{
    full = b >= lo && b + 8 <= hi;
    float sq[8];
    const uint64_t inv2 = f2(inv, inv);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        f2_split(f2_mul(f2(s[2 * q], s[2 * q + 1]), inv2), gv[2 * q], gv[2 * q + 1]);
        sq[2 * q] = gv[2 * q];
        sq[2 * q + 1] = gv[2 * q + 1];
    }
    in = 0xffu;
    if (b + 8 > psi || !full) {  // padding, or a group cut by the tile/window edge
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint64_t i = b + e;
            if (i >= psi)
                gv[e] = 0.0f;
            if (!(i >= lo && i < hi))
                in &= ~(1u << e);
            sq[e] = (in >> e & 1u) ? gv[e] : 0.0f;
        }
    }
    if (squares_in_range(sq)) {  // every counted element finite: no overflow
        const uint64_t scale2 = f2(kSqScale, kSqScale);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            acc.add_pair(f2_mul(f2(sq[2 * q], sq[2 * q + 1]), scale2));
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            bad |= (in >> e & 1u) && not_finite(gv[e]);
        acc.wide += sumsq_wide(gv[0], gv[1], gv[2], gv[3], gv[4], gv[5], gv[6], gv[7], in);
    }
}

/* One warp's share of a tile's sum of squares: its fp32 pair and its rare fp64 part. */
struct WarpPart {
    float h, l;
    double wide;
};

/* A tile's sum of squares from every thread's accumulator: a fixed-order pair-arithmetic
 * shuffle tree in fp32 per warp, then the kThreads / 32 warp pairs pairwise in the same
 * arithmetic, ((w0 + w4) + (w2 + w6)) + ((w1 + w5) + (w3 + w7)) for 8 warps, and fp64
 * once per tile: GB300's fp64 pipe is a small fraction of its fp32 rate, and at N = 2 a
 * conversion per warp kept it a third busy.  The fp64 parts of the rare out-of-range
 * groups (zero almost always, tested with integer compares) are added in the same tree
 * shape.  The warp values alternate between two buffers (`parity`), so a following tile
 * cannot overwrite them before thread 0 has read them.  Called by the block's first
 * kThreads threads only, which meet at named barrier 1 (other warps of a larger block go
 * on unhindered).  The result is valid in thread 0 only. */
template <int kThreads>
__device__ __forceinline__ double tile_fold(const SumSq& acc, WarpPart (*warp_part)[kThreads / 32],
                                            uint32_t& parity)
{
    constexpr int W = kThreads / 32;
    static_assert(W <= 32 && (W & (W - 1)) == 0, "warp tree");
    float ph, pl, h1, l1;
    f2_split(acc.hi2, ph, h1);
    f2_split(acc.lo2, pl, l1);
    pair_add(ph, pl, h1, l1);  // the even elements' pair + the odd elements' pair
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float h2 = __shfl_xor_sync(0xffffffffu, ph, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, pl, o);
        pair_add(ph, pl, h2, l2);
    }
    double wide = acc.wide;  // >= 0: any set bit means nonzero
    if (__any_sync(0xffffffffu, __double_as_longlong(wide) != 0)) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            wide += __shfl_xor_sync(0xffffffffu, wide, o);
    }
    WarpPart* wp = warp_part[parity];
    const int lane = threadIdx.x & 31;
    if (lane == 0)
        wp[threadIdx.x >> 5] = WarpPart{ph, pl, wide};
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
    double t = 0.0;
    if (threadIdx.x == 0) {
        float h[W], l[W];
        long long any_wide = 0;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            h[w] = wp[w].h;
            l[w] = wp[w].l;
            any_wide |= __double_as_longlong(wp[w].wide);
        }
        // pairwise: independent pair additions, three levels deep for 8 warps
#pragma unroll
        for (int hh = W / 2; hh > 0; hh >>= 1)
#pragma unroll
            for (int w = 0; w < hh; ++w)
                pair_add(h[w], l[w], h[w + hh], l[w + hh]);
        t = ((double)h[0] + (double)l[0]) * kSqUnscale;
        if (any_wide != 0) {
            double x[W];
#pragma unroll
            for (int w = 0; w < W; ++w)
                x[w] = wp[w].wide;
#pragma unroll
            for (int hh = W / 2; hh > 0; hh >>= 1)
#pragma unroll
                for (int w = 0; w < hh; ++w)
                    x[w] = x[w] + x[w + hh];
            t += x[0];
        }
    }
    parity ^= 1u;
    return t;
}

}  // namespace
}  // namespace zero
