/*
 * adamw_elem.cuh -- the AdamW element update and the bulk-copy ring helpers shared by the
 * AdamW kernels (adamw.cu: state in HBM; adamw_variants.cu: the re-reading schedule and
 * the state in host memory), so every variant computes the same bits.
 *
 * Per element, in fp32 and in this order (the _rn intrinsics forbid FMA contraction, so
 * the result is the correctly rounded value of each written operation):
 *   gc = c*g;  m = b1*m + (1-b1)*gc;  v = b2*v + (1-b2)*(gc*gc)
 *   p  = p*decay - step_size * (m / (sqrt(v)/rbc2 + eps));  out = bf16_rne(p) (or fp16)
 */
#pragma once

#include "zero_internal.h"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

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

/* Two gathered parameters, rounded to nearest even, in one 32-bit word (lo first). */
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    if (F16) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

template <bool F16>
__device__ __forceinline__ uint16_t pack1(float x)
{
    return F16 ? __half_as_ushort(__float2half_rn(x)) : __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

/* Wait for phase `parity` of an mbarrier, at most ~2 s (4e9 cycles); 0 on timeout. */
__device__ __forceinline__ uint32_t wait_parity_bounded(uint32_t bar, uint32_t parity)
{
    const long long t0 = clock64();
    uint32_t ok = 0;
    while (true) {
        asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
                     "selp.u32 %0, 1, 0, p; }"
                     : "=r"(ok)
                     : "r"(bar), "r"(parity)
                     : "memory");
        if (ok || clock64() - t0 > 4000000000LL)
            return ok;
    }
}

/* One bulk copy global -> shared (`bytes` a multiple of 16, both addresses 16-byte
 * aligned), completing on the mbarrier at shared address `bar`.  With EvictFirst the copy
 * carries an L2 policy that marks what it brings in as first to evict: every byte the
 * AdamW passes read is read exactly once, so on buffers many times larger than L2 it then
 * keeps the lines being written (master, m, v and the parameters leave through L2) in
 * preference to inputs already consumed.  Measured on the GPT-2-1.5B buffer: k_adamw
 * 6.87 -> 6.68 ms (1.00 -> 1.03 of the copy peak), and the next step's reduce 4.54 ->
 * 4.38 ms; on buffers of 2^22-2^25 parameters the same policy cost 1-3%, so the launchers
 * pick the kernel by size (adamw_evict_first).  A compile-time choice: a run-time flag
 * tested in the copy-issuing path cost ~2 us per step by itself. */
template <bool EvictFirst>
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    if constexpr (EvictFirst) {
        uint64_t pol;
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
                     "[%0], [%1], %2, [%3], %4;"
                     ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(pol)
                     : "memory");
    } else {
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
                     "[%0], [%1], %2, [%3];"
                     ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                     : "memory");
    }
}

constexpr int kChunk = 4096;  // elements per bulk-copied chunk of each array
constexpr int kStages = 3;
constexpr size_t kSmemBytes = (size_t)kStages * 4 * kChunk * sizeof(float);  // 192 KiB
constexpr uint64_t kNoChunk = ~0ull;  // a ring stage with no chunk: the chunk queue is empty

}  // namespace
}  // namespace zero
