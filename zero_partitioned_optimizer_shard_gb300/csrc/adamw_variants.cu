/*
 * adamw_variants.cu -- the fused AdamW + cast + gathered write of adamw.cu in two other
 * data placements, with the same element arithmetic (adamw_elem.cuh):
 *   - k_adamw_rereduce: the re-reading schedule at N = 2 (g formed again from the two
 *     gradient copies instead of read from a materialised fp32 g);
 *   - k_adamw_host_state: master, m and v in page-locked host memory, updated in place
 *     over the CPU-GPU link.
 */
#include "adamw_elem.cuh"

#include <atomic>

namespace zero {
namespace {

/*
 * The re-reading schedule for N = 2.  Clipping needs the global norm before any update,
 * so an exact step either writes the fp32 g and reads it back (34 + 2N bytes per
 * parameter) or reads the N gradient copies twice (26 + 4N): at N = 2 that is 34 instead
 * of 38 B.  The reduce pass then stores no g (only the tile sums of squares and the
 * overflow flag), and this kernel forms each g[i] again from the two copies with the
 * reduce's arithmetic, (0 + x0[i]) + x1[i] in fp32 times the step's f32(1/(N*L)), so the
 * update is bit-identical.  Same ring as k_adamw: per stage the two 4096-element copy
 * chunks (8 KiB each) take the place of g's 16 KiB.
 */
template <zero_dtype_t DT>
__device__ __forceinline__ float grad_value(uint16_t b)
{
    return DT == ZERO_F16 ? __half2float(__ushort_as_half(b)) : __uint_as_float((uint32_t)b << 16);
}

template <zero_dtype_t DT>
__device__ __forceinline__ float regather(uint16_t x0, uint16_t x1, float inv)
{
    return __fmul_rn(__fadd_rn(__fadd_rn(0.0f, grad_value<DT>(x0)), grad_value<DT>(x1)), inv);
}

template <zero_dtype_t DT, bool F16, bool EF>
__global__ void __launch_bounds__(kBlock, 1) k_adamw_rereduce(const __grid_constant__ AdamwArgs a)
{
    extern __shared__ __align__(128) float ring[];  // kStages x {x0|x1, master, m, v} x kChunk
    __shared__ __align__(8) uint64_t full[kStages];
    __shared__ uint64_t s_chunk[kStages];  // the chunk each stage holds, or kNoChunk
    grid_dependency_wait();
    const zero_step_state_t* st = a.st;
    if (st->skip)
        return;
    __shared__ Scalars s_sh;
    __shared__ float s_inv;
    if (threadIdx.x == 0) {
        s_sh.c = st->clip_coef;
        s_sh.step = st->step_size;
        s_sh.rbc2 = st->rbc2;
        s_sh.decay = st->decay;
        s_sh.b1 = a.beta1;
        s_sh.b2 = a.beta2;
        s_sh.omb1 = __fsub_rn(1.0f, a.beta1);
        s_sh.omb2 = __fsub_rn(1.0f, a.beta2);
        s_sh.eps = a.eps;
        s_inv = st->inv_scale_used;
    }
    __syncthreads();
    const Scalars& s = s_sh;
    const float inv = s_inv;

    const uint64_t n_chunks = a.psi / kChunk;

    if (threadIdx.x == 0) {
        for (int k = 0; k < kStages; ++k)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&full[k])));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // chunks from the step state's queue, as in k_adamw: stage k gets chunk c (its index
    // published by the barrier's arrival), or, past the last chunk, an arrival alone
    auto issue = [&](int k, uint64_t c) {
        const uint32_t bar = smem_addr(&full[k]);
        if (c >= n_chunks) {
            s_chunk[k] = kNoChunk;
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
            return;
        }
        s_chunk[k] = c;
        const uint64_t base = c * (uint64_t)kChunk;
        float* stage = ring + k * 4 * kChunk;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                     ::"r"(bar), "r"((uint32_t)(4 * kChunk * sizeof(float))) : "memory");
        const void* src[5] = {a.rep0 + base, a.rep1 + base, a.master + base, a.m + base, a.v + base};
        const uint32_t bytes[5] = {kChunk * 2, kChunk * 2, kChunk * 4, kChunk * 4, kChunk * 4};
        float* dst[5] = {stage, stage + kChunk / 2, stage + kChunk, stage + 2 * kChunk,
                         stage + 3 * kChunk};
        for (int q = 0; q < 5; ++q)
            bulk_load<EF>(smem_addr(dst[q]), src[q], bytes[q], bar);
    };
    uint64_t ahead = 0;  // thread 0: the next chunk it will issue
    if (threadIdx.x == 0) {
        for (int k = 0; k < kStages; ++k)
            issue(k, atomicAdd(a.next_chunk, 1ull));
        ahead = atomicAdd(a.next_chunk, 1ull);
    }

    bool failed = false;
    for (uint64_t i = 0;; ++i) {
        const int k = (int)(i % kStages);
        const uint32_t ok = wait_parity_bounded(smem_addr(&full[k]), (uint32_t)((i / kStages) & 1));
        if (__syncthreads_or(!ok)) {  // the whole block leaves the ring together
            if (threadIdx.x == 0) {
                atomicOr(a.err, 1u);
                for (uint64_t j = i; j < i + kStages; ++j)  // every stage was issued
                    wait_parity_bounded(smem_addr(&full[j % kStages]), (uint32_t)((j / kStages) & 1));
            }
            failed = true;
            break;
        }
        const uint64_t c = s_chunk[k];
        if (c == kNoChunk)  // the queue ran dry: every later stage is empty too
            break;
        const float* stage = ring + k * 4 * kChunk;
        const uint16_t* s0 = reinterpret_cast<const uint16_t*>(stage);
        const uint16_t* s1 = reinterpret_cast<const uint16_t*>(stage + kChunk / 2);
        const float* sp = stage + kChunk;
        const float* sm = stage + 2 * kChunk;
        const float* sv = stage + 3 * kChunk;
        const uint64_t base = c * (uint64_t)kChunk;
#pragma unroll
        for (int e = threadIdx.x * 4; e < kChunk; e += kBlock * 4) {
            const uint2 x0 = *reinterpret_cast<const uint2*>(s0 + e);
            const uint2 x1 = *reinterpret_cast<const uint2*>(s1 + e);
            float4 p0 = *reinterpret_cast<const float4*>(sp + e);
            float4 m0 = *reinterpret_cast<const float4*>(sm + e);
            float4 v0 = *reinterpret_cast<const float4*>(sv + e);
            const float g0 = regather<DT>((uint16_t)(x0.x & 0xffffu), (uint16_t)(x1.x & 0xffffu), inv);
            const float g1 = regather<DT>((uint16_t)(x0.x >> 16), (uint16_t)(x1.x >> 16), inv);
            const float g2 = regather<DT>((uint16_t)(x0.y & 0xffffu), (uint16_t)(x1.y & 0xffffu), inv);
            const float g3 = regather<DT>((uint16_t)(x0.y >> 16), (uint16_t)(x1.y >> 16), inv);
            uint2 o;
            o.x = pack2<F16>(adamw_one(g0, p0.x, m0.x, v0.x, s), adamw_one(g1, p0.y, m0.y, v0.y, s));
            o.y = pack2<F16>(adamw_one(g2, p0.z, m0.z, v0.z, s), adamw_one(g3, p0.w, m0.w, v0.w, s));
            __stcs(reinterpret_cast<float4*>(a.master + base + e), p0);
            __stcs(reinterpret_cast<float4*>(a.m + base + e), m0);
            __stcs(reinterpret_cast<float4*>(a.v + base + e), v0);
            __stcs(reinterpret_cast<uint2*>(a.out + base + e), o);
        }
        __syncthreads();  // stage k fully read (and s_chunk[k] by every thread): refill it
        if (threadIdx.x == 0) {
            issue(k, ahead);
            if (ahead < n_chunks)
                ahead = atomicAdd(a.next_chunk, 1ull);
        }
    }

    const uint64_t stride = (uint64_t)gridDim.x * kBlock;
    const uint64_t tid = (uint64_t)blockIdx.x * kBlock + threadIdx.x;
    for (uint64_t i = n_chunks * kChunk + tid; !failed && i < a.psi_padded; i += stride) {
        if (i < a.psi) {
            float p = a.master[i], m = a.m[i], v = a.v[i];
            const float r = adamw_one(regather<DT>(a.rep0[i], a.rep1[i], inv), p, m, v, s);
            a.master[i] = p;
            a.m[i] = m;
            a.v[i] = v;
            a.out[i] = pack1<F16>(r);
        } else {
            a.out[i] = 0;
        }
    }
    // the queue back to 0 for the next launch, by the last block to finish
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(a.done, 1u) == gridDim.x - 1) {
            __threadfence();
            atomicExch(a.next_chunk, 0ull);
            atomicExch(a.done, 0u);
        }
    }
}

/*
 * The same update with master, m and v resident in pinned host memory ("ZeRO 显存优化"
 * sec. 6: the optimizer state may be offloaded to the CPU, at a transfer cost to be
 * measured on the machine).  On GB300 the Grace host memory is reached over NVLink-C2C
 * by ordinary loads and stores, so the step stays one fused kernel: each element's state
 * crosses the link once in each direction (12 B up, 12 B down) while g is read from and
 * the gathered parameter written to HBM.  The link, not HBM, bounds it; the kernel keeps
 * enough 128-bit loads in flight per thread (two groups of four elements from each of
 * the four arrays) to cover the link's latency.  Bulk-copy rings are not used for host
 * memory: plain loads measured the link's full rate.  The arithmetic is adamw_one,
 * so results are bit-identical to k_adamw's.
 */
constexpr int kHostUnroll = 2;

template <bool F16>
__global__ void __launch_bounds__(kBlock) k_adamw_host_state(const __grid_constant__ AdamwArgs a)
{
    grid_dependency_wait();
    const zero_step_state_t* st = a.st;
    if (st->skip)
        return;
    __shared__ Scalars s_sh;
    if (threadIdx.x == 0) {
        s_sh.c = st->clip_coef;
        s_sh.step = st->step_size;
        s_sh.rbc2 = st->rbc2;
        s_sh.decay = st->decay;
        s_sh.b1 = a.beta1;
        s_sh.b2 = a.beta2;
        s_sh.omb1 = __fsub_rn(1.0f, a.beta1);
        s_sh.omb2 = __fsub_rn(1.0f, a.beta2);
        s_sh.eps = a.eps;
    }
    __syncthreads();
    const Scalars& s = s_sh;

    const uint64_t n4 = a.psi / 4;  // whole groups of four, none holding padding
    const uint64_t stride = (uint64_t)gridDim.x * kBlock;
    const uint64_t tid = (uint64_t)blockIdx.x * kBlock + threadIdx.x;
    const float4* g4 = reinterpret_cast<const float4*>(a.g);
    float4* p4 = reinterpret_cast<float4*>(a.master);
    float4* m4 = reinterpret_cast<float4*>(a.m);
    float4* v4 = reinterpret_cast<float4*>(a.v);
    uint2* o4 = reinterpret_cast<uint2*>(a.out);
    for (uint64_t j = tid; j < n4; j += kHostUnroll * stride) {
        float4 g[kHostUnroll], p[kHostUnroll], m[kHostUnroll], v[kHostUnroll];
#pragma unroll
        for (int u = 0; u < kHostUnroll; ++u) {
            const uint64_t q = j + u * stride;
            if (q < n4) {
                g[u] = __ldcs(g4 + q);
                p[u] = __ldcs(p4 + q);
                m[u] = __ldcs(m4 + q);
                v[u] = __ldcs(v4 + q);
            }
        }
#pragma unroll
        for (int u = 0; u < kHostUnroll; ++u) {
            const uint64_t q = j + u * stride;
            if (q < n4) {
                uint2 o;
                o.x = pack2<F16>(adamw_one(g[u].x, p[u].x, m[u].x, v[u].x, s),
                                 adamw_one(g[u].y, p[u].y, m[u].y, v[u].y, s));
                o.y = pack2<F16>(adamw_one(g[u].z, p[u].z, m[u].z, v[u].z, s),
                                 adamw_one(g[u].w, p[u].w, m[u].w, v[u].w, s));
                __stcs(p4 + q, p[u]);
                __stcs(m4 + q, m[u]);
                __stcs(v4 + q, v[u]);
                __stcs(o4 + q, o);
            }
        }
    }
    for (uint64_t i = n4 * 4 + tid; i < a.psi_padded; i += stride) {
        if (i < a.psi) {
            float p = a.master[i], m = a.m[i], v = a.v[i];
            const float r = adamw_one(a.g[i], p, m, v, s);
            a.master[i] = p;
            a.m[i] = m;
            a.v[i] = v;
            a.out[i] = pack1<F16>(r);
        } else {
            a.out[i] = 0;
        }
    }
}

}  // namespace

template <bool EF>
cudaError_t launch_rereduce_ef(const AdamwArgs& a, dim3 g, dim3 b, cudaStream_t s)
{
    if (a.grad_f16)
        return a.out_f16 ? launch_pdl(k_adamw_rereduce<ZERO_F16, true, EF>, g, b, kSmemBytes, s, a)
                         : launch_pdl(k_adamw_rereduce<ZERO_F16, false, EF>, g, b, kSmemBytes, s, a);
    return a.out_f16 ? launch_pdl(k_adamw_rereduce<ZERO_BF16, true, EF>, g, b, kSmemBytes, s, a)
                     : launch_pdl(k_adamw_rereduce<ZERO_BF16, false, EF>, g, b, kSmemBytes, s, a);
}

cudaError_t launch_adamw_rereduce(const AdamwArgs& a, cudaStream_t s)
{
    // the kernel takes its chunks from the step state's queue and writes through these
    if (!a.next_chunk || !a.done || !a.err || !a.rep0 || !a.rep1)
        return cudaErrorInvalidValue;
    static std::atomic<bool> configured[64];  // per device; a race only repeats the set-up
    int dev = 0;
    cudaGetDevice(&dev);
    if (!configured[dev & 63].load(std::memory_order_relaxed)) {
        for (auto kern : {k_adamw_rereduce<ZERO_BF16, false, false>, k_adamw_rereduce<ZERO_BF16, true, false>,
                          k_adamw_rereduce<ZERO_F16, false, false>, k_adamw_rereduce<ZERO_F16, true, false>,
                          k_adamw_rereduce<ZERO_BF16, false, true>, k_adamw_rereduce<ZERO_BF16, true, true>,
                          k_adamw_rereduce<ZERO_F16, false, true>, k_adamw_rereduce<ZERO_F16, true, true>}) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)kSmemBytes);
            if (e != cudaSuccess)
                return e;
        }
        configured[dev & 63].store(true, std::memory_order_relaxed);
    }
    const uint64_t chunks = a.psi / kChunk;
    const uint64_t tail_blocks = (a.psi_padded - chunks * kChunk + kBlock - 1) / kBlock;
    const uint64_t want = chunks > tail_blocks ? chunks : tail_blocks;
    const uint64_t cap = (uint64_t)sm_count();
    const dim3 g((unsigned)(want < cap ? (want > 0 ? want : 1) : cap)), b(kBlock);
    return adamw_evict_first(a.psi_padded, 30) ? launch_rereduce_ef<true>(a, g, b, s)
                                               : launch_rereduce_ef<false>(a, g, b, s);
}

cudaError_t launch_adamw_host_state(const AdamwArgs& a, cudaStream_t s)
{
    const uint64_t groups = a.psi / 4;
    const uint64_t tail = a.psi_padded - groups * 4;
    const uint64_t want_threads = (groups + kHostUnroll - 1) / kHostUnroll;
    uint64_t want = ((want_threads > tail ? want_threads : tail) + kBlock - 1) / kBlock;
    const uint64_t cap = (uint64_t)sm_count() * 3;  // 80 registers x 256 threads: 3 blocks per SM
    const unsigned grid = (unsigned)(want < cap ? (want > 0 ? want : 1) : cap);
    return a.out_f16 ? launch_pdl(k_adamw_host_state<true>, dim3(grid), dim3(kBlock), 0, s, a)
                     : launch_pdl(k_adamw_host_state<false>, dim3(grid), dim3(kBlock), 0, s, a);
}

}  // namespace zero
