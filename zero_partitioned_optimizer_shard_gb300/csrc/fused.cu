/*
 * fused.cu -- the whole step in one launch for small layouts (k_step_fused).
 *
 * Below a few million parameters the three-launch step (reduce, norm, AdamW) is bound by
 * latency, not bandwidth: each launch costs a few microseconds of ramp-up and drain, the
 * norm kernel's chain of fp64 operations sits between the other two, and the fp32
 * gradient makes a round trip through memory.  When every tile of the layout can have a
 * block resident at the same time, one cooperative launch does it all:
 *
 *   1. block u takes tile u of the sum-of-squares grid (a shard cut at the flat multiples
 *      of 8192, as in the reduce pass) and forms g there with the reduce pass's own
 *      arithmetic and thread-to-element mapping (reduce_elem.cuh), so g and the tile's
 *      partial come out with the same bits; g stays in shared memory (and is written to
 *      the caller's g buffer when one is given);
 *   2. the block stores its tile partial, ORs its overflow flag and arrives on the
 *      launch's counter; the last block to arrive forms the global norm from the
 *      partials in the norm kernel's order (one warp per rank, the rank's slots
 *      lane-strided, a fixed shuffle tree, ranks in order; the order finalize.cu uses for
 *      layouts of at most 128 tiles per rank) and the clip coefficient, and releases
 *      the other blocks with one 64-bit store (the counter back to 0, the step's c or -1
 *      for a skipped step) as soon as that outcome is certain (for c = 1, often from an
 *      upward-rounded fp32 bound of the sum, before the exact norm); it zeroes the
 *      partials and applies the skip decision and loss scaler to the state
 *      (step_scalars.cuh); every block forms the step's other scalars (bias
 *      corrections, decay) itself;
 *   3. every block applies AdamW to its tile from the g it holds (adamw_elem.cuh) and
 *      writes the gathered parameters.  Master, m and v were fetched while step 1 ran:
 *      into shared memory by bulk copies when the layout has at most one tile per SM
 *      (the staged shape, 17 warps), else into L2 by prefetches (9 warps, 3 blocks/SM).
 *      In the staged shape the 9 warps that do not stream have already updated the tile
 *      with c = 1 while the norm was formed (master, m, v and the gathered parameters
 *      written through to global memory, the shared-memory copies of master, m, v and of
 *      the gathered parameters as found kept); a block whose step has c = 1 (c = 1
 *      multiplies g exactly: the same bits) has only its tile's few edge elements left;
 *      with another c it updates again from the copies, and if the step does not apply
 *      it puts everything back from them.
 *
 * So the results are bit-identical to the three-launch step, and the traffic is
 * 2N + 26 bytes per parameter (+4 when g is written; staged, +2 for reading the gathered
 * parameters as found), not 2N + 34.  "【论文解读】ZeRO"
 * sec. 6(2) describes the same three stages per rank (reduce-scatter, shard update,
 * all-gather); only their scheduling differs.
 *
 * Waiting: the launch is cooperative (every block resident at once), and a block that
 * waits for the last one gives up after ~2 s, records 1 in the step state's error word and
 * writes nothing more.  GB300's fp64 arithmetic is slow (64 cycles per dependent add,
 * about 650 per division or square root), so the fp64 chains that need no norm run in
 * warps of their own beside the streaming ones: the bias corrections of step t+1 and, in
 * the staged shape, the loss scaler's two possible outcomes; only the streaming warps
 * meet before the arrival (named barriers).
 */
#include "adamw_elem.cuh"
#include "reduce_elem.cuh"
#include "step_scalars.cuh"

#include <atomic>

namespace zero {
namespace {

#ifdef ZERO_TEST_HOOKS
/* Test builds only (never the product library): the bounded-wait test names one block
 * that leaves without arriving, so the other blocks' wait for the last one runs out
 * without any fault. */
__device__ unsigned long long zero_test_absent_block = ~0ull;
#endif

constexpr int kFusedWarps = 8;                       // stream the gradients (phase 1)
constexpr int kFusedThreads = kFusedWarps * 32;      // the reduce pass's block size
constexpr int kFusedLoads = 8;                       // replica loads in flight per thread (N <= 8)
constexpr int kFusedLoadsWide = 16;                  // N > 8: the N = 16 and the generic kernel
constexpr uint64_t kT = ZERO_TILE_ELEMS;
constexpr int kGcFloats = (int)kT + 8;               // the tile's g from its first whole group

static_assert(kFusedThreads == 256, "the tile partial's bits depend on the reduce pass's block size");

/* Two shapes of the same kernel.  Unstaged: 9 warps (8 streaming, 1 for the scalar chains),
 * up to 3 blocks per SM, master/m/v prefetched into L2.  Staged, for layouts of at most one
 * tile per SM: 17 warps (the 8 streaming ones, 8 more, the scalar warp); the tile's master,
 * m and v are bulk-copied into shared memory when the block starts, and the 9 other warps
 * update the tile speculatively with c = 1 from there while the streaming warps fold,
 * arrive and wait for the norm. */
template <bool STAGED>
struct Shape {
    static constexpr int kScalarWarp = STAGED ? 16 : 8;
    static constexpr int kThreads = (kScalarWarp + 1) * 32;
    static constexpr int kMinBlocks = STAGED ? 1 : 3;
    // named barrier 5: the streaming warps wait there for the warps that read the state
    // and form the step's scalars (the scalar warp; staged also warp 8)
    static constexpr int kScalarsReady = kFusedThreads + 32 * (STAGED ? 2 : 1);
    // g (+ master, m, v and the speculative gathered parameters)
    static constexpr size_t kSmem = (size_t)kGcFloats * 4 * (STAGED ? 4 : 1) + (STAGED ? (size_t)kGcFloats * 2 : 0);
};

/* The launch's 64-bit word: the state's launch_arrivals (low half, the arrival counter)
 * and applied_c (high half, the step's outcome).  Arrival: acquire-release, so this
 * block's writes are ordered before it and the last block to arrive sees every block's
 * writes. */
__device__ __forceinline__ uint64_t arrive_acq_rel(uint64_t* p)
{
    uint64_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u64 %0, [%1], 1;" : "=l"(old) : "l"(p) : "memory");
    return old;
}

/* The release and the wait for it: relaxed, single 64-bit accesses.  A waiting block
 * takes nothing from the last block but the word itself (its other scalars are its own,
 * its tile is disjoint from every other), so nothing needs ordering around them. */
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

/* True only when the clip coefficient min(1, max_norm / (norm + 1e-6)) of the exact fp64
 * computation (clip_coefficient of the fp64 sum of the partials) is certainly 1, judged
 * from u >= the exact sum of the partials, formed in fp32 with upward rounding.  With
 * b = RU(sqrt(u)) >= sqrt(sum), the fp64 path's rounded sum exceeds the exact one by less
 * than 2^-45 relatively, its square root and its + 1e-6 round up by 2^-53 at most, so its
 * divisor is at most (b (1 + 2^-45) + 1e-6)(1 + 2^-53) < the bound formed here; a divisor
 * <= max_norm gives a quotient >= 1, which stays >= 1 when rounded, so c = 1. */
__device__ __forceinline__ bool clip_certainly_one(float u, float max_norm)
{
    const float b = __fsqrt_ru(u);
    const float need = __fmul_ru(__fadd_ru(__fmul_ru(b, 1.000001f), 1.0000001e-6f), 1.000001f);
    return max_norm >= need;
}

/* L2 prefetch of the bytes [p, p + n), rounded inwards to 16-byte boundaries (a hint:
 * the data is read with ordinary loads later). */
__device__ __forceinline__ void prefetch_l2(const void* p, uint64_t n)
{
    const uintptr_t a0 = ((uintptr_t)p + 15u) & ~(uintptr_t)15u;
    const uintptr_t a1 = ((uintptr_t)p + n) & ~(uintptr_t)15u;
    if (a1 > a0)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                     ::"l"(a0), "r"((uint32_t)(a1 - a0)) : "memory");
}

/* Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) into shared
 * memory, completing on the mbarrier `bar`. */
__device__ __forceinline__ void bulk_to_smem(void* dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

/* AdamW of one element i < psi, or the padding's gathered 0; [lo, hi) is the block's tile. */
__device__ __forceinline__ void update_one(const FusedArgs& a, uint64_t i, float g, const Scalars& s,
                                           uint64_t lo, uint64_t hi)
{
    if (!ZERO_OWNED(i, 1, lo, hi, &a.st->error))
        return;
    if (i < a.psi) {
        float p = a.master[i], m = a.m[i], v = a.v[i];
        const float r = adamw_one(g, p, m, v, s);
        a.master[i] = p;
        a.m[i] = m;
        a.v[i] = v;
        a.out[i] = a.out_f16 ? pack1<true>(r) : pack1<false>(r);
    } else {
        a.out[i] = 0;
    }
}

template <zero_dtype_t DT, int NR, bool STAGED>
__global__ void __launch_bounds__(Shape<STAGED>::kThreads, NR == 0 && !STAGED ? 2 : Shape<STAGED>::kMinBlocks)
k_step_fused(const __grid_constant__ FusedArgs a)
{
    using S = Shape<STAGED>;
    extern __shared__ __align__(16) float dyn[];  // g of the tile; staged: then master, m, v
    float* const gc = dyn;                        // gc[i - base] holds g[i]
    __shared__ WarpPart warp_part[2][kFusedWarps];
    __shared__ double rank_sum[ZERO_MAX_KERNEL_RANKS];
    __shared__ float rank_up[kFusedWarps];  // an upward-rounded fp32 bound of each rank's sum
    __shared__ float s_step, s_rbc2, s_decay;
    __shared__ float s_applied;  // the step's outcome: c, or -1 when the step is skipped
    __shared__ ScalerCand s_cand;  // staged: the scaler's outcomes, formed ahead of time
    __shared__ Scalars s_sc;
    __shared__ __align__(16) zero_step_state_t s_st;  // the state as this step found it
    __shared__ __align__(8) uint64_t s_bar;            // staged: the bulk copies
    __shared__ uint32_t s_flag;  // last block; then: released (or last)
    __shared__ uint32_t s_spec;  // staged: the bulk copies landed and the speculation ran
    grid_launch_dependents();
    grid_dependency_wait();
    zero_step_state_t* st = a.st;
    uint64_t* const word = reinterpret_cast<uint64_t*>(&st->launch_arrivals);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t N = NR > 0 ? (uint32_t)NR : a.n_ranks;
    const float inv = st->inv_scale;

    // this block's tile: slot u = r * tiles_per_rank + j
    const uint64_t u = blockIdx.x, tpr = a.tiles_per_rank;
    const uint64_t r = u / tpr, j = u - r * tpr;
    const uint64_t shard_lo = r * a.shard, shard_hi = shard_lo + a.shard;
    const uint64_t cell = (shard_lo / kT + j) * kT;
    const uint64_t lo = cell > shard_lo ? cell : shard_lo;
    const uint64_t hi = cell + kT < shard_hi ? cell + kT : shard_hi;
    const uint64_t base = lo & ~7ull;                           // first group of the tile
    const uint64_t v_lo = (lo + 3) & ~3ull, v_hi = hi & ~3ull;  // 16-byte-aligned body
    const bool staged_copy = STAGED && lo < hi && v_lo < v_hi;
    float* const sp = dyn + kGcFloats;  // staged master, m, v, indexed like gc
    float* const sm = sp + kGcFloats;
    float* const sv = sm + kGcFloats;
    const uint32_t bar = smem_addr(&s_bar);

    if (threadIdx.x == 0) {
        s_spec = 0;
        s_applied = -1.0f;
    }
    if (staged_copy && threadIdx.x == 0) {
        // the tile's optimizer state into shared memory, in flight while the gradients are
        // summed; only the 16-byte-aligned body, the few edge elements are read directly
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        const uint32_t bytes = (uint32_t)((v_hi - v_lo) * sizeof(float));
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                     ::"r"(bar), "r"(3 * bytes) : "memory");
        bulk_to_smem(sp + (v_lo - base), a.master + v_lo, bytes, bar);
        bulk_to_smem(sm + (v_lo - base), a.m + v_lo, bytes, bar);
        bulk_to_smem(sv + (v_lo - base), a.v + v_lo, bytes, bar);
    }
    if (w == S::kScalarWarp) {
        // a copy of the state for the last block, and the bias corrections of step t+1
        // (lanes 0 and 1 run the two fp64 power chains side by side); all read before this
        // block arrives (barrier 5), so before the last block rewrites the state
        if (lane < (int)(sizeof(zero_step_state_t) / 16))
            reinterpret_cast<uint4*>(&s_st)[lane] = __ldcg(reinterpret_cast<const uint4*>(st) + lane);
        if (lane < 2) {
            const uint32_t t_next = st->t + 1;
            if (lane == 0)
                s_step = bias_step_size(a.hp, t_next);
            else
                s_rbc2 = bias_rbc2(a.hp, t_next);
        }
        if (lane == 3)
            s_decay = decoupled_decay(a.hp);
        if (!STAGED && lane == 2 && lo < hi) {
            prefetch_l2(a.master + lo, (hi - lo) * sizeof(float));
            prefetch_l2(a.m + lo, (hi - lo) * sizeof(float));
            prefetch_l2(a.v + lo, (hi - lo) * sizeof(float));
        }
        __syncwarp();
        asm volatile("bar.arrive 5, %0;" ::"n"(S::kScalarsReady) : "memory");
    }
    if (STAGED && w == kFusedWarps) {
        // a warp that is idle until the AdamW phase forms the scaler's two outcomes (two
        // fp64 divisions) for the last block
        if (lane == 0) {
            const zero_step_state_t s0 = *st;
            s_cand = scaler_candidates(s0, a.hp, N);
        }
        __syncwarp();
        asm volatile("bar.arrive 5, %0;" ::"n"(S::kScalarsReady) : "memory");
    }

    // 1. g over the tile: the reduce pass's groups and order; several groups' loads in
    // flight per thread before their ordered sums
    SumSq acc;
    bool bad = false;
    if (w < kFusedWarps && lo < hi) {
        constexpr int GB = NR > 0 && NR < kFusedLoads ? kFusedLoads / NR : 1;  // groups per batch
        constexpr int LB = NR > 0 && NR <= kFusedLoads ? kFusedLoads : kFusedLoadsWide;  // loads per batch
        for (uint64_t b0 = base + 8ull * threadIdx.x; b0 < hi; b0 += 8ull * kFusedThreads * GB) {
            uint4 v[GB][NR > 0 && NR < kFusedLoads ? NR : LB];
            if (NR > 0 && NR < kFusedLoads) {
#pragma unroll
                for (int q = 0; q < GB; ++q) {
                    const uint64_t b = b0 + 8ull * kFusedThreads * q;
                    if (b < hi && b + 8 <= a.psi_padded) {
#pragma unroll
                        for (int k = 0; k < (NR > 0 ? NR : 1); ++k)
                            v[q][k] = ld_stream_v4((const uint16_t*)a.rep[k] + b);
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < GB; ++q) {
                const uint64_t b = b0 + 8ull * kFusedThreads * q;
                if (b >= hi)
                    break;
                float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                if (b + 8 <= a.psi_padded) {
                    if (NR > 0 && NR < kFusedLoads) {
#pragma unroll
                        for (int k = 0; k < (NR > 0 ? NR : 1); ++k)
                            add8<DT>(s, v[q][k]);
                    } else {
#pragma unroll 1
                        for (uint32_t k0 = 0; k0 < N; k0 += LB) {
#pragma unroll
                            for (int kk = 0; kk < LB; ++kk)
                                if (k0 + kk < N)
                                    v[0][kk] = ld_stream_v4((const uint16_t*)a.rep[k0 + kk] + b);
#pragma unroll
                            for (int kk = 0; kk < LB; ++kk)
                                if (k0 + kk < N)
                                    add8<DT>(s, v[0][kk]);
                        }
                    }
                } else {  // the buffer's last, ragged group: element loads inside the tile
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const uint64_t i = b + e;
                        if (i >= lo && i < hi)
                            for (uint32_t k = 0; k < N; ++k)
                                s[e] = __fadd_rn(s[e], one16<DT>(ld_stream_u16((const uint16_t*)a.rep[k] + i)));
                    }
                }
                float gv[8];
                uint32_t in;
                bool full;
                group_values(a.psi, inv, s, b, lo, hi, acc, bad, gv, in, full);
                float* c = gc + (b - base);
                if (full) {
                    if (ZERO_OWNED(b - base, 8, 0, kGcFloats, &st->error)) {
                        *reinterpret_cast<float4*>(c) = make_float4(gv[0], gv[1], gv[2], gv[3]);
                        *reinterpret_cast<float4*>(c + 4) = make_float4(gv[4], gv[5], gv[6], gv[7]);
                    }
                    if (a.g && ZERO_OWNED(b, 8, lo, hi, &st->error)) {
                        __stcs(reinterpret_cast<float4*>(a.g + b), make_float4(gv[0], gv[1], gv[2], gv[3]));
                        __stcs(reinterpret_cast<float4*>(a.g + b + 4), make_float4(gv[4], gv[5], gv[6], gv[7]));
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (in >> e & 1u) {
                            if (ZERO_OWNED(b + e - base, 1, 0, kGcFloats, &st->error))
                                c[e] = gv[e];
                            if (a.g && ZERO_OWNED(b + e, 1, lo, hi, &st->error))
                                a.g[b + e] = gv[e];
                        }
                }
            }
        }
    }

    // staged: g of the tile is ready for the warps that only update (named barrier 3:
    // the streaming warps arrive, the others wait)
    if (STAGED && w < kFusedWarps)
        asm volatile("bar.arrive 3, %0;" ::"n"(S::kThreads) : "memory");

    // 2. the tile's partial (the reduce pass's fold), the overflow flag, and arrival: only
    // the streaming warps meet here (named barriers), so the other warps' fp64 chains and
    // the staged speculation below do not hold the arrival or the norm back
    if (w < kFusedWarps) {
        uint32_t parity = 0;
        const double part = tile_fold<kFusedThreads>(acc, warp_part, parity);
        if (threadIdx.x == 0 && lo < hi)
            __stcg(a.partials + u, part);
        if (__any_sync(0xffffffffu, bad) && lane == 0)
            atomicOr(&st->overflow, 1u);
        // before this block arrives, its scalar warps have read the state (which the last
        // block rewrites once every block has arrived) and formed the scalars the last
        // block uses
        asm volatile("bar.sync 5, %0;" ::"n"(S::kScalarsReady) : "memory");
        if (threadIdx.x == 0) {
#ifdef ZERO_TEST_HOOKS
            if (blockIdx.x == zero_test_absent_block)
                s_flag = 2;  // test builds only: this block never arrives
            else
#endif
            s_flag = (uint32_t)arrive_acq_rel(word) == gridDim.x - 1;
        }
        asm volatile("bar.sync 2, %0;" ::"n"(kFusedThreads) : "memory");

        if (s_flag == 1) {
            // the last block: the norm in the norm kernel's order (at most 128 slots per
            // rank: lane l adds slots l, l+32, l+64, l+96 in that order), partials zeroed;
            // thread 0 fetches the overflow flag meanwhile.  The others are released as
            // soon as their outcome is certain: at once for a skipped step, and, with at
            // most one rank per warp, before the exact norm when an fp32 upper bound of
            // the sum already shows c = 1 (clip_certainly_one); the exact norm, c and the
            // state follow.
            constexpr bool kEarly = NR > 0 && NR <= kFusedWarps;
            uint32_t overflow = 0;
            bool released = false;  // thread 0
            if (threadIdx.x == 0)
                overflow = __ldcg(&st->overflow) != 0;
            auto release = [&](float applied) {
                // the counter back to 0 and the outcome, in one store
                st_relaxed_u64(word, (uint64_t)__float_as_uint(applied) << 32);
                s_applied = applied;
                released = true;
            };
            auto rank_sum_of = [&](uint32_t rr, const double (&v)[4]) {
                double* p = a.partials + (uint64_t)rr * tpr;
                double s = 0.0;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint64_t c = lane + 32u * q;
                    if (c < tpr) {
                        s += v[q];
                        p[c] = 0.0;
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    s += __shfl_xor_sync(0xffffffffu, s, o);
                if (lane == 0)
                    rank_sum[rr] = s;
            };
            auto load_rank = [&](uint32_t rr, double (&v)[4]) {
                const double* p = a.partials + (uint64_t)rr * tpr;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint64_t c = lane + 32u * q;
                    v[q] = c < tpr ? __ldcg(p + c) : 0.0;
                }
            };
            if (kEarly) {
                double v[4];
                if ((uint32_t)w < N) {
                    load_rank(w, v);
                    float up = 0.0f;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        up = __fadd_ru(up, __double2float_ru(v[q]));
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
                        up = __fadd_ru(up, __shfl_xor_sync(0xffffffffu, up, o));
                    if (lane == 0)
                        rank_up[w] = up;
                }
                asm volatile("bar.sync 2, %0;" ::"n"(kFusedThreads) : "memory");
                if (threadIdx.x == 0) {
                    if (overflow) {
                        release(-1.0f);
                    } else if (!(a.hp.max_grad_norm > 0.0f)) {
                        release(1.0f);  // clipping disabled
                    } else {
                        float u = 0.0f;
                        for (uint32_t rr = 0; rr < N; ++rr)
                            u = __fadd_ru(u, rank_up[rr]);
                        if (clip_certainly_one(u, a.hp.max_grad_norm))
                            release(1.0f);
                    }
                }
                if ((uint32_t)w < N)
                    rank_sum_of(w, v);
            } else {
                if (threadIdx.x == 0 && overflow)
                    release(-1.0f);
                for (uint32_t rr = w; rr < N; rr += kFusedWarps) {
                    double v[4];
                    load_rank(rr, v);
                    rank_sum_of(rr, v);
                }
            }
            asm volatile("bar.sync 2, %0;" ::"n"(kFusedThreads) : "memory");
            if (threadIdx.x == 0) {
                double total = 0.0;
                for (uint32_t rr = 0; rr < N; ++rr)
                    total += rank_sum[rr];
                const double norm = sqrt(total);
                // released already: a skipped step or a certain c = 1 (no fp64 division)
                const float c = released ? 1.0f : clip_coefficient(norm, overflow, a.hp.max_grad_norm);
                const float applied = overflow ? -1.0f : c;
                if (!released)
                    release(applied);
                // the state for the next step, read after the launch: every field the step
                // changes, never the error word (other blocks may still OR into it), the
                // launch word (written above) or what the step leaves as it is
                zero_step_state_t& ls = s_st;
                const uint32_t t_next = ls.t + 1;
                if (!overflow) {
                    ls.step_size = s_step;
                    ls.rbc2 = s_rbc2;
                }
                if (STAGED)
                    scaler_apply(&ls, s_cand, overflow, t_next);
                else
                    scaler_update(&ls, a.hp, N, overflow, t_next);
                ls.sumsq = total;
                ls.norm = norm;
                ls.clip_coef = c;
                ls.overflow = 0;
                ls.n_steps += 1;
                ls.applied_c = applied;
                static_assert(offsetof(zero_step_state_t, n_ranks) == 64, "fields [0, 64) in four stores");
                for (int q = 0; q < 4; ++q)
                    __stcg(reinterpret_cast<uint4*>(st) + q, reinterpret_cast<const uint4*>(&ls)[q]);
                __stcg(&st->n_steps, ls.n_steps);
                __stcg(&st->n_skipped, ls.n_skipped);
                __stcg(&st->inv_scale_used, ls.inv_scale_used);
            }
        } else if (s_flag == 0 && threadIdx.x == 0) {
            // wait for the last block's release, at most ~2 s
            const long long t0 = clock64();
            uint32_t ok = 1;
            uint64_t wv;
            while ((uint32_t)(wv = ld_relaxed_u64(word)) != 0) {
                if (clock64() - t0 > 4000000000LL) {
                    ok = 0;
                    atomicOr(&st->error, 1u);
                    break;
                }
                __nanosleep(64);
            }
            s_applied = __uint_as_float((uint32_t)(wv >> 32));
            s_flag = ok;
        }
        if (threadIdx.x == 0) {
            // the update's scalars: the released c and this block's own step t + 1 scalars
            // (the same bits as the last block's: same inputs, same arithmetic)
            s_sc.c = s_applied;
            s_sc.step = s_step;
            s_sc.rbc2 = s_rbc2;
            s_sc.decay = s_decay;
            s_sc.b1 = a.hp.beta1;
            s_sc.b2 = a.hp.beta2;
            s_sc.omb1 = __fsub_rn(1.0f, a.hp.beta1);
            s_sc.omb2 = __fsub_rn(1.0f, a.hp.beta2);
            s_sc.eps = a.hp.eps;
        }
    } else if (STAGED && staged_copy) {
        // staged: meanwhile the other warps update the tile speculatively with c = 1 (the
        // step's other scalars need no norm) from the shared-memory copies of master, m
        // and v, which stay as they are.  The new master, m, v and gathered parameters go
        // straight to global memory, so their writing overlaps the wait for the norm.
        // c = 1 multiplies g exactly, so if the step's clip coefficient turns out to be 1
        // these are the step's bits; if not they are made again with the real c, and if
        // the step does not apply they are undone, both from the shared-memory copies (the
        // gathered parameters as the step found them are kept for that too: each thread
        // loads the 4-element groups it will update while the gradients are summed)
        constexpr int kSpec = S::kThreads - kFusedThreads;
        constexpr int kOutGroups = (int)((kT / 4 + kSpec - 1) / kSpec);
        const int t = threadIdx.x - kFusedThreads;
        static_assert(4 * kOutGroups * kSpec >= (int)kT, "every group of a tile has a slot");
        const uint64_t v_end = v_hi < (a.psi & ~3ull) ? v_hi : (a.psi & ~3ull);  // may be < v_lo
        uint16_t* const so = reinterpret_cast<uint16_t*>(sv + kGcFloats);
        {
            uint2 o0[kOutGroups];
#pragma unroll
            for (int q = 0; q < kOutGroups; ++q) {
                const uint64_t i = v_lo + 4ull * (t + q * kSpec);
                if (i < v_end)
                    o0[q] = __ldcs(reinterpret_cast<const uint2*>(a.out + i));
            }
#pragma unroll
            for (int q = 0; q < kOutGroups; ++q) {
                const uint64_t i = v_lo + 4ull * (t + q * kSpec);
                if (i < v_end && ZERO_OWNED(i - base, 4, 0, kGcFloats, &st->error))
                    *reinterpret_cast<uint2*>(so + (i - base)) = o0[q];
            }
        }
        asm volatile("bar.sync 3, %0;" ::"n"(S::kThreads) : "memory");
        if (t == 0) {
            s_spec = wait_parity_bounded(bar, 0);
            if (!s_spec)
                atomicOr(&st->error, 1u);
        }
        asm volatile("bar.sync 4, %0;" ::"n"(S::kThreads - kFusedThreads) : "memory");
        if (s_spec) {
            Scalars sc;
            sc.c = 1.0f;
            sc.step = s_step;
            sc.rbc2 = s_rbc2;
            sc.decay = s_cand.decay;
            sc.b1 = a.hp.beta1;
            sc.b2 = a.hp.beta2;
            sc.omb1 = __fsub_rn(1.0f, a.hp.beta1);
            sc.omb2 = __fsub_rn(1.0f, a.hp.beta2);
            sc.eps = a.hp.eps;
            for (uint64_t i = v_lo + 4ull * t; i < v_end; i += 4ull * kSpec) {
                const uint64_t k = i - base;
                const float4 g4 = *reinterpret_cast<const float4*>(gc + k);
                float4 p4 = *reinterpret_cast<const float4*>(sp + k);
                float4 m4 = *reinterpret_cast<const float4*>(sm + k);
                float4 v4 = *reinterpret_cast<const float4*>(sv + k);
                uint2 o;
                if (a.out_f16) {
                    o.x = pack2<true>(adamw_one(g4.x, p4.x, m4.x, v4.x, sc), adamw_one(g4.y, p4.y, m4.y, v4.y, sc));
                    o.y = pack2<true>(adamw_one(g4.z, p4.z, m4.z, v4.z, sc), adamw_one(g4.w, p4.w, m4.w, v4.w, sc));
                } else {
                    o.x = pack2<false>(adamw_one(g4.x, p4.x, m4.x, v4.x, sc), adamw_one(g4.y, p4.y, m4.y, v4.y, sc));
                    o.y = pack2<false>(adamw_one(g4.z, p4.z, m4.z, v4.z, sc), adamw_one(g4.w, p4.w, m4.w, v4.w, sc));
                }
                if (ZERO_OWNED(i, 4, lo, hi, &st->error)) {
                    __stcs(reinterpret_cast<float4*>(a.master + i), p4);
                    __stcs(reinterpret_cast<float4*>(a.m + i), m4);
                    __stcs(reinterpret_cast<float4*>(a.v + i), v4);
                    __stcs(reinterpret_cast<uint2*>(a.out + i), o);
                }
            }
        }
    } else if (STAGED) {
        asm volatile("bar.sync 3, %0;" ::"n"(S::kThreads) : "memory");
    }
    __syncthreads();

    // 3. AdamW over the tile, unless the step is skipped or this block gave up waiting.
    // Staged, after the speculative update (already written with c = 1): with c = 1 only
    // the edge elements remain; with another c the tile is updated again from the
    // shared-memory copies; if the step does not apply here, master, m, v and the gathered
    // parameters are put back from them.  Otherwise the update reads master, m, v from global memory.
    // Every thread derives the same mode from the shared flags:
    // 0 nothing; 1 speculation kept (only the tile's edges remain); 2 update again from the
    // shared-memory copies; 3 update from global memory; 4 undo the speculation (put
    // master, m, v and the gathered parameters back)
    const bool go = s_flag == 1 && !(__float_as_uint(s_applied) >> 31) && lo < hi;
    const bool copy_failed = STAGED && staged_copy && !s_spec;  // error recorded: write nothing
    uint32_t mode = 0;
    if (STAGED && staged_copy && s_spec)
        mode = !go ? 4 : s_applied == 1.0f ? 1 : 2;
    else if (go && !copy_failed)
        mode = 3;
    const bool edges = go && !copy_failed;
    {
        const Scalars& sc = s_sc;
        // [v_lo, v_end): whole 4-element groups below psi; [v_end, v_hi): the group holding
        // psi and the padding (v_end is never below v_lo: a tile that starts past psi has
        // no vector part)
        uint64_t v_end = v_hi < (a.psi & ~3ull) ? v_hi : (a.psi & ~3ull);
        v_end = v_end > v_lo ? v_end : v_lo;
        if (edges) {
            if (v_lo >= v_hi) {
                for (uint64_t i = lo + threadIdx.x; i < hi; i += S::kThreads)
                    update_one(a, i, gc[i - base], sc, lo, hi);
            } else {
                if (lo + threadIdx.x < v_lo)
                    update_one(a, lo + threadIdx.x, gc[lo + threadIdx.x - base], sc, lo, hi);
                if (v_hi + threadIdx.x < hi)
                    update_one(a, v_hi + threadIdx.x, gc[v_hi + threadIdx.x - base], sc, lo, hi);
                // the groups holding psi or padding, element by element
                for (uint64_t i = v_end + 4ull * threadIdx.x; i < v_hi; i += 4ull * S::kThreads)
                    for (int e = 0; e < 4; ++e)
                        update_one(a, i + e, gc[i + e - base], sc, lo, hi);
            }
        }
        // mode 1: the speculation wrote the tile's vector part already
        if (mode == 4) {
            const uint16_t* const so = reinterpret_cast<const uint16_t*>(sv + kGcFloats);
            for (uint64_t i = v_lo + 4ull * threadIdx.x; i < v_end; i += 4ull * S::kThreads) {
                const uint64_t k = i - base;
                if (!ZERO_OWNED(i, 4, lo, hi, &st->error))
                    continue;
                __stcs(reinterpret_cast<float4*>(a.master + i), *reinterpret_cast<const float4*>(sp + k));
                __stcs(reinterpret_cast<float4*>(a.m + i), *reinterpret_cast<const float4*>(sm + k));
                __stcs(reinterpret_cast<float4*>(a.v + i), *reinterpret_cast<const float4*>(sv + k));
                __stcs(reinterpret_cast<uint2*>(a.out + i), *reinterpret_cast<const uint2*>(so + k));
            }
        } else if (mode == 2 || mode == 3) {
            // Q 4-element groups per thread at a time: all their loads before any store
            // (the arrays may alias as far as the compiler knows, so it would not hoist
            // them itself)
            constexpr int Q = 3;
            for (uint64_t i0 = v_lo + 4ull * threadIdx.x; i0 < v_end; i0 += 4ull * S::kThreads * Q) {
                float4 p4[Q], m4[Q], v4[Q];
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    const uint64_t i = i0 + 4ull * S::kThreads * q;
                    if (i < v_end) {
                        if (STAGED && mode == 2) {
                            p4[q] = *reinterpret_cast<const float4*>(sp + (i - base));
                            m4[q] = *reinterpret_cast<const float4*>(sm + (i - base));
                            v4[q] = *reinterpret_cast<const float4*>(sv + (i - base));
                        } else {
                            p4[q] = __ldcs(reinterpret_cast<const float4*>(a.master + i));
                            m4[q] = __ldcs(reinterpret_cast<const float4*>(a.m + i));
                            v4[q] = __ldcs(reinterpret_cast<const float4*>(a.v + i));
                        }
                    }
                }
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    const uint64_t i = i0 + 4ull * S::kThreads * q;
                    if (i >= v_end)
                        break;
                    const float4 g4 = *reinterpret_cast<const float4*>(gc + (i - base));
                    uint2 o;
                    if (a.out_f16) {
                        o.x = pack2<true>(adamw_one(g4.x, p4[q].x, m4[q].x, v4[q].x, sc),
                                          adamw_one(g4.y, p4[q].y, m4[q].y, v4[q].y, sc));
                        o.y = pack2<true>(adamw_one(g4.z, p4[q].z, m4[q].z, v4[q].z, sc),
                                          adamw_one(g4.w, p4[q].w, m4[q].w, v4[q].w, sc));
                    } else {
                        o.x = pack2<false>(adamw_one(g4.x, p4[q].x, m4[q].x, v4[q].x, sc),
                                           adamw_one(g4.y, p4[q].y, m4[q].y, v4[q].y, sc));
                        o.y = pack2<false>(adamw_one(g4.z, p4[q].z, m4[q].z, v4[q].z, sc),
                                           adamw_one(g4.w, p4[q].w, m4[q].w, v4[q].w, sc));
                    }
                    if (!ZERO_OWNED(i, 4, lo, hi, &st->error))
                        continue;
                    __stcs(reinterpret_cast<float4*>(a.master + i), p4[q]);
                    __stcs(reinterpret_cast<float4*>(a.m + i), m4[q]);
                    __stcs(reinterpret_cast<float4*>(a.v + i), v4[q]);
                    __stcs(reinterpret_cast<uint2*>(a.out + i), o);
                }
            }
        }
    }
    // staged: the bulk copies land in this block's shared memory; never leave before they
    // have (bounded), whatever the path taken above
    if (staged_copy && threadIdx.x == 0 && !s_spec && !wait_parity_bounded(bar, 0))
        atomicOr(&st->error, 1u);
}

template <zero_dtype_t DT, int NR, bool STAGED>
struct FusedKernel {
    static constexpr auto kernel = k_step_fused<DT, NR, STAGED>;
    using S = Shape<STAGED>;
    static int capacity()  // blocks that can be resident at once, cached per device
    {
        static std::atomic<int> cap[64];  // per device; a race only repeats the query
        int dev = 0;
        cudaGetDevice(&dev);
        int c = cap[dev & 63].load(std::memory_order_relaxed);
        if (c == 0) {
            int o = 0;
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)S::kSmem) == cudaSuccess)
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kernel, S::kThreads, S::kSmem);
            cudaGetLastError();  // a refused attribute or query leaves no error behind
            c = o > 0 ? o * sm_count() : -1;
            cap[dev & 63].store(c, std::memory_order_relaxed);
        }
        return c;
    }
    static cudaError_t launch(const FusedArgs& a, unsigned grid, cudaStream_t s)
    {
        // cooperative (all blocks resident together) and, where the driver accepts the
        // pair, programmatic dependent launch; the choice is remembered per device
        static std::atomic<int> mode[64];  // 0 unknown, 1 both attributes, 2 cooperative only
        int dev = 0;
        cudaGetDevice(&dev);
        std::atomic<int>& md = mode[dev & 63];
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(S::kThreads);
        cfg.dynamicSmemBytes = S::kSmem;
        cfg.stream = s;
        cudaLaunchAttribute at[2];
        at[0].id = cudaLaunchAttributeCooperative;
        at[0].val.cooperative = 1;
        at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        if (md != 2) {
            cfg.numAttrs = 2;
            cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a);
            if (e == cudaSuccess) {
                md = 1;
                return e;
            }
            if (md == 1 || e == cudaErrorCooperativeLaunchTooLarge)
                return e;  // not about the pair of attributes
            cudaGetLastError();  // the pair was refused: clear it, use cooperative alone
            md = 2;
        }
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kernel, a);
    }
};

template <zero_dtype_t DT, bool STAGED>
int capacity_dt(uint32_t n)
{
    switch (n) {
    case 2: return FusedKernel<DT, 2, STAGED>::capacity();
    case 4: return FusedKernel<DT, 4, STAGED>::capacity();
    case 8: return FusedKernel<DT, 8, STAGED>::capacity();
    case 16: return FusedKernel<DT, 16, STAGED>::capacity();
    default: return FusedKernel<DT, 0, STAGED>::capacity();
    }
}

template <zero_dtype_t DT, bool STAGED>
cudaError_t launch_dt(const FusedArgs& a, unsigned grid, cudaStream_t s)
{
    switch (a.n_ranks) {
    case 2: return FusedKernel<DT, 2, STAGED>::launch(a, grid, s);
    case 4: return FusedKernel<DT, 4, STAGED>::launch(a, grid, s);
    case 8: return FusedKernel<DT, 8, STAGED>::launch(a, grid, s);
    case 16: return FusedKernel<DT, 16, STAGED>::launch(a, grid, s);
    default: return FusedKernel<DT, 0, STAGED>::launch(a, grid, s);
    }
}

}  // namespace

#ifdef ZERO_TEST_HOOKS
extern "C" int zero_test_absent_fused_block(unsigned long long block)
{
    return cudaMemcpyToSymbol(zero_test_absent_block, &block, sizeof block) == cudaSuccess ? 0 : -4;
}
#endif

int fused_shape(const zero_layout_t* L, zero_dtype_t dtype)
{
    if (L->n_buckets != 1 || L->tiles_per_rank > kFusedMaxTilesPerRank)
        return 0;
    const bool f16 = dtype == ZERO_F16;
    const int staged = f16 ? capacity_dt<ZERO_F16, true>(L->n_ranks) : capacity_dt<ZERO_BF16, true>(L->n_ranks);
    if (staged > 0 && L->n_tiles <= (uint64_t)staged)
        return 2;
    const int plain = f16 ? capacity_dt<ZERO_F16, false>(L->n_ranks) : capacity_dt<ZERO_BF16, false>(L->n_ranks);
    return plain > 0 && L->n_tiles <= (uint64_t)plain ? 1 : 0;
}

cudaError_t launch_step_fused(const FusedArgs& a, zero_dtype_t dtype, uint64_t n_tiles, int shape,
                              cudaStream_t s)
{
    const unsigned grid = (unsigned)n_tiles;
    if (dtype == ZERO_F16)
        return shape == 2 ? launch_dt<ZERO_F16, true>(a, grid, s) : launch_dt<ZERO_F16, false>(a, grid, s);
    return shape == 2 ? launch_dt<ZERO_BF16, true>(a, grid, s) : launch_dt<ZERO_BF16, false>(a, grid, s);
}

}  // namespace zero
