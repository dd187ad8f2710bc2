/*
 * adamw.cu -- fused AdamW on the fp32 master/momentum/variance shards + bf16 gather.
 *
 * "【论文解读】ZeRO" sec. 6(2): after the reduce-scatter each rank updates only its own
 * partition with its own reduced gradient, and the all-gather rebuilds the full parameter
 * vector [p0' ... p7'] with every shard at its own offset.  Writing rank r's bf16 result
 * at flat [r*S, (r+1)*S) of one buffer is that gathered layout; with all ranks on this GPU
 * one pass over the flat index updates every shard.  The optimizer is AdamW (operatorworld
 * ZeRO article and the Megatron page name it; the update is Adam with bias correction and
 * decoupled weight decay), fp32 state, bf16 parameters.
 *
 * Per element, in fp32 and in this order (the _rn intrinsics forbid FMA contraction, so
 * the result is the correctly rounded value of each written operation):
 *   gc = c*g;  m = b1*m + (1-b1)*gc;  v = b2*v + (1-b2)*(gc*gc)
 *   p  = p*decay - step_size * (m / (sqrt(v)/rbc2 + eps));  out = bf16_rne(p)
 * c, step_size, rbc2 and decay come from the step state written by the norm kernel; a
 * skipped step (overflow) leaves every byte untouched.
 *
 * GB300 design: HBM streaming, 16 bytes read and 14 written per element.  A persistent
 * grid-stride loop moves 8 elements per thread per iteration: two 128-bit loads from each
 * of g (non-coherent, L1 bypass), master, m, v (streaming), two 128-bit streaming stores
 * to each of master, m, v and one 128-bit store of 8 bf16 parameters.
 */
#include "zero_internal.h"

#include <cuda_bf16.h>

namespace zero {
namespace {

constexpr int kBlock = 256;

struct Scalars {
    float c, step, rbc2, decay, b1, b2, omb1, omb2, eps;
};

__device__ __forceinline__ float adamw_one(float g, float& p, float& m, float& v, const Scalars& s)
{
    const float gc = __fmul_rn(s.c, g);
    m = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, gc));
    v = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(s.omb2, __fmul_rn(gc, gc)));
    const float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), s.rbc2), s.eps);
    p = __fsub_rn(__fmul_rn(p, s.decay), __fmul_rn(s.step, __fdiv_rn(m, denom)));
    return p;
}

__device__ __forceinline__ float4 ld_nc_v4(const float* p)
{
    float4 v;
    asm("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(kBlock) k_adamw(const __grid_constant__ AdamwArgs a)
{
    const zero_step_state_t* st = a.st;
    if (st->skip)
        return;
    Scalars s;
    s.c = st->clip_coef;
    s.step = st->step_size;
    s.rbc2 = st->rbc2;
    s.decay = st->decay;
    s.b1 = a.beta1;
    s.b2 = a.beta2;
    s.omb1 = __fsub_rn(1.0f, a.beta1);
    s.omb2 = __fsub_rn(1.0f, a.beta2);
    s.eps = a.eps;

    const uint64_t stride = (uint64_t)gridDim.x * kBlock;
    const uint64_t tid = (uint64_t)blockIdx.x * kBlock + threadIdx.x;
    const uint64_t n_full = a.psi / 8;  // groups of 8 with no padding

    for (uint64_t q = tid; q < n_full; q += stride) {
        const uint64_t b = q * 8;
        const float4 g0 = ld_nc_v4(a.g + b), g1 = ld_nc_v4(a.g + b + 4);
        float4 p0 = __ldcs(reinterpret_cast<const float4*>(a.master + b));
        float4 p1 = __ldcs(reinterpret_cast<const float4*>(a.master + b + 4));
        float4 m0 = __ldcs(reinterpret_cast<const float4*>(a.m + b));
        float4 m1 = __ldcs(reinterpret_cast<const float4*>(a.m + b + 4));
        float4 v0 = __ldcs(reinterpret_cast<const float4*>(a.v + b));
        float4 v1 = __ldcs(reinterpret_cast<const float4*>(a.v + b + 4));
        uint4 o;
        o.x = pack_bf16x2(adamw_one(g0.x, p0.x, m0.x, v0.x, s), adamw_one(g0.y, p0.y, m0.y, v0.y, s));
        o.y = pack_bf16x2(adamw_one(g0.z, p0.z, m0.z, v0.z, s), adamw_one(g0.w, p0.w, m0.w, v0.w, s));
        o.z = pack_bf16x2(adamw_one(g1.x, p1.x, m1.x, v1.x, s), adamw_one(g1.y, p1.y, m1.y, v1.y, s));
        o.w = pack_bf16x2(adamw_one(g1.z, p1.z, m1.z, v1.z, s), adamw_one(g1.w, p1.w, m1.w, v1.w, s));
        __stcs(reinterpret_cast<float4*>(a.master + b), p0);
        __stcs(reinterpret_cast<float4*>(a.master + b + 4), p1);
        __stcs(reinterpret_cast<float4*>(a.m + b), m0);
        __stcs(reinterpret_cast<float4*>(a.m + b + 4), m1);
        __stcs(reinterpret_cast<float4*>(a.v + b), v0);
        __stcs(reinterpret_cast<float4*>(a.v + b + 4), v1);
        __stcs(reinterpret_cast<uint4*>(a.out + b), o);
    }

    // the ragged end: the group holding psi, and whole padding groups up to psi_padded
    const uint64_t n_groups = (a.psi_padded + 7) / 8;
    for (uint64_t q = n_full + tid; q < n_groups; q += stride) {
        for (int e = 0; e < 8; ++e) {
            const uint64_t i = q * 8 + e;
            if (i >= a.psi_padded)
                break;
            if (i < a.psi) {
                float p = a.master[i], m = a.m[i], v = a.v[i];
                const float r = adamw_one(a.g[i], p, m, v, s);
                a.master[i] = p;
                a.m[i] = m;
                a.v[i] = v;
                a.out[i] = __bfloat16_as_ushort(__float2bfloat16_rn(r));
            } else {
                a.out[i] = 0;  // padding: gathered value 0, state untouched
            }
        }
    }
}

}  // namespace

cudaError_t launch_adamw(const AdamwArgs& a, cudaStream_t s)
{
    static int per_sm[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    int& occ = per_sm[dev & 63];
    if (occ == 0) {
        int o = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, k_adamw, kBlock, 0);
        occ = o > 0 ? o : 1;
    }
    const uint64_t groups = (a.psi_padded + 7) / 8;
    const uint64_t want = (groups + kBlock - 1) / kBlock;
    const uint64_t cap = (uint64_t)sm_count() * (uint64_t)occ;
    const unsigned grid = (unsigned)(want < cap ? want : cap);
    k_adamw<<<grid > 0 ? grid : 1, kBlock, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace zero
