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
 * skipped step (overflow) leaves every byte untouched.  The gathered parameters are bf16,
 * or fp16 when asked (the FP16 replicated parameters of "【论文解读】ZeRO" sec. 4(1)).
 *
 * GB300 design: HBM streaming, 16 bytes read and 14 written per element.  The inputs
 * are staged by the Blackwell bulk-copy engine: one thread per block issues
 * cp.async.bulk copies of 4096-element chunks of g, master, m and v (64 KiB per chunk)
 * into a three-stage shared-memory ring tracked by mbarriers, so up to 192 KiB per SM are
 * in flight without holding registers.  On buffers many times larger than L2 the copies
 * carry an L2 evict-first policy (each input byte is read once), which keeps L2 for the
 * lines being written.  One 256-thread block per SM (persistent, taking its chunks in
 * order from a queue in the step state) computes from shared memory and writes master,
 * m, v and 8 bf16 parameters per thread with streaming 128/64-bit stores.  The ragged end (the part
 * after the last whole chunk, and the padding) is done element by element.  Every
 * mbarrier wait is bounded (~2 s); on a timeout the block records an error in the step
 * state, waits (bounded) for its copies in flight and leaves.
 */
#include "adamw_elem.cuh"

#include <atomic>

namespace zero {
namespace {

#ifdef ZERO_TEST_HOOKS
/* Test builds only (never the product library): the bounded-wait test names one chunk
 * whose copies are withheld, so that chunk's mbarrier wait runs out without any fault. */
__device__ unsigned long long zero_test_withheld_chunk = ~0ull;
#endif

template <bool F16, bool EF>
__global__ void __launch_bounds__(kBlock, 1) k_adamw(const __grid_constant__ AdamwArgs a)
{
    extern __shared__ __align__(128) float ring[];  // kStages x {g, master, m, v} x kChunk
    __shared__ __align__(8) uint64_t full[kStages];
    __shared__ uint64_t s_chunk[kStages];  // the chunk each stage holds, or kNoChunk
    grid_dependency_wait();
    const zero_step_state_t* st = a.st;
    if (st->skip)
        return;
    // the step's scalars live in shared memory: held in registers they cost the unrolled
    // element loop about 10% (measured), from register pressure in the fp32 division chains
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

    const uint64_t n_chunks = a.psi / kChunk;  // whole chunks, none holding padding
    const float* src[4] = {a.g, a.master, a.m, a.v};

    if (threadIdx.x == 0) {
        for (int k = 0; k < kStages; ++k)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&full[k])));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // Stage k gets chunk c: its index for the block (published by the barrier's arrival),
    // then the four bulk copies; past the last chunk, an arrival with no copies.
    auto issue = [&](int k, uint64_t c) {
        const uint32_t bar = smem_addr(&full[k]);
        if (c >= n_chunks) {
            s_chunk[k] = kNoChunk;
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
            return;
        }
        s_chunk[k] = c;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                     ::"r"(bar), "r"((uint32_t)(4 * kChunk * sizeof(float))) : "memory");
#ifdef ZERO_TEST_HOOKS
        if (c == zero_test_withheld_chunk)
            return;  // test builds only: this chunk's barrier never completes
#endif
        for (int q = 0; q < 4; ++q)
            bulk_load<EF>(smem_addr(ring + (k * 4 + q) * kChunk), src[q] + c * kChunk,
                          (uint32_t)(kChunk * sizeof(float)), bar);
    };
    // Chunks are handed out in order by one counter in the step state, one at a time to
    // the block that asks: the chunks in flight stay together at the front of the buffers
    // however the blocks' speeds differ, and a faster block takes more of them.  (A fixed
    // assignment, block b taking chunks b, b + gridDim.x, ..., let the blocks drift apart
    // over long launches: 0.999 of the copy peak on the Llama-7B buffer in one launch,
    // 1.031 in four.)  Thread 0 takes each chunk one refill ahead of its use, so the
    // atomic's latency stays off the ring's path.
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
        const float* sg = ring + (k * 4 + 0) * kChunk;
        const float* sp = ring + (k * 4 + 1) * kChunk;
        const float* sm = ring + (k * 4 + 2) * kChunk;
        const float* sv = ring + (k * 4 + 3) * kChunk;
        const uint64_t base = c * (uint64_t)kChunk;
#pragma unroll
        for (int e = threadIdx.x * 4; e < kChunk; e += kBlock * 4) {
            const float4 g0 = *reinterpret_cast<const float4*>(sg + e);
            float4 p0 = *reinterpret_cast<const float4*>(sp + e);
            float4 m0 = *reinterpret_cast<const float4*>(sm + e);
            float4 v0 = *reinterpret_cast<const float4*>(sv + e);
            uint2 o;
            o.x = pack2<F16>(adamw_one(g0.x, p0.x, m0.x, v0.x, s), adamw_one(g0.y, p0.y, m0.y, v0.y, s));
            o.y = pack2<F16>(adamw_one(g0.z, p0.z, m0.z, v0.z, s), adamw_one(g0.w, p0.w, m0.w, v0.w, s));
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

    // the ragged end: after the last whole chunk, up to psi_padded (padding gets out = 0)
    const uint64_t stride = (uint64_t)gridDim.x * kBlock;
    const uint64_t tid = (uint64_t)blockIdx.x * kBlock + threadIdx.x;
    for (uint64_t i = n_chunks * kChunk + tid; !failed && i < a.psi_padded; i += stride) {
        if (i < a.psi) {
            float p = a.master[i], m = a.m[i], v = a.v[i];
            const float r = adamw_one(a.g[i], p, m, v, s);
            a.master[i] = p;
            a.m[i] = m;
            a.v[i] = v;
            a.out[i] = pack1<F16>(r);
        } else {
            a.out[i] = 0;  // padding: gathered value 0, state untouched
        }
    }
    // the queue back to 0 for the next launch, by the last block to finish (every block
    // has taken its last chunk before it counts itself done)
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(a.done, 1u) == gridDim.x - 1) {
            __threadfence();
            atomicExch(a.next_chunk, 0ull);
            atomicExch(a.done, 0u);
        }
    }
}

}  // namespace

#ifdef ZERO_TEST_HOOKS
extern "C" int zero_test_withhold_adamw_chunk(unsigned long long chunk)
{
    return cudaMemcpyToSymbol(zero_test_withheld_chunk, &chunk, sizeof chunk) == cudaSuccess ? 0 : -4;
}
#endif

cudaError_t launch_adamw(const AdamwArgs& a, cudaStream_t s)
{
    // the kernel takes its chunks from the step state's queue and writes through these
    if (!a.next_chunk || !a.done || !a.err)
        return cudaErrorInvalidValue;
    static std::atomic<bool> configured[64];  // per device; a race only repeats the set-up
    int dev = 0;
    cudaGetDevice(&dev);
    if (!configured[dev & 63].load(std::memory_order_relaxed)) {
        for (auto kern : {k_adamw<false, false>, k_adamw<true, false>, k_adamw<false, true>,
                          k_adamw<true, true>}) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)kSmemBytes);
            if (e != cudaSuccess)
                return e;
        }
        configured[dev & 63].store(true, std::memory_order_relaxed);
    }
    const bool ef = adamw_evict_first(a.psi_padded, 30);
    const uint64_t chunks = a.psi / kChunk;
    const uint64_t tail_blocks = (a.psi_padded - chunks * kChunk + kBlock - 1) / kBlock;
    const uint64_t want = chunks > tail_blocks ? chunks : tail_blocks;
    const uint64_t cap = (uint64_t)sm_count();  // one 192 KiB block per SM
    const unsigned grid = (unsigned)(want < cap ? want : cap);
    const dim3 g(grid > 0 ? grid : 1), b(kBlock);
    if (ef)
        return a.out_f16 ? launch_pdl(k_adamw<true, true>, g, b, kSmemBytes, s, a)
                         : launch_pdl(k_adamw<false, true>, g, b, kSmemBytes, s, a);
    return a.out_f16 ? launch_pdl(k_adamw<true, false>, g, b, kSmemBytes, s, a)
                     : launch_pdl(k_adamw<false, false>, g, b, kSmemBytes, s, a);
}

}  // namespace zero
