/*
 * partition.cu -- zero_partition and zero_workspace_bytes: host-only integer layout.
 *
 * "【论文解读】ZeRO" sec. 4(1)-(3): the model states are divided into N_d equal partitions
 * and data-parallel rank i keeps and updates partition i.  A flat buffer of Psi elements
 * is cut into N shards of S = ceil(Psi/N) elements (rounded up to `align`); the buffer
 * is padded to N*S so every shard has the same length and rank r's starts at r*S.
 *
 * Ledger (same page sec. 2(1) and 8; "ZeRO 显存优化" sec. 3): 2 bytes of fp16/bf16
 * weight, 2 of gradient and K = 12 of fp32 master/momentum/variance per parameter.  Plain
 * DP keeps 16*Psi; stage 1 keeps full weights and gradients and a 12-byte shard; stage 2
 * keeps full weights and a 14-byte shard; stage 3 keeps only a 16-byte shard.  Counted on
 * the allocated (padded) buffers.  Communication ("【论文解读】ZeRO" sec. 6(1)-(3)): a ring
 * reduce-scatter or all-gather sends (N-1) chunks of S per rank; plain DP and stages 1-2
 * send two of them per step, stage 3 three.
 */
#include "zero_internal.h"

#include <string.h>

extern "C" int zero_partition(uint64_t psi, uint32_t n_ranks, uint32_t stage, uint32_t align,
                              uint64_t bucket_elems, zero_layout_t* out)
{
    if (!out || psi == 0 || psi > (1ull << 56) || n_ranks == 0 || n_ranks > ZERO_MAX_RANKS ||
        stage > 3 || align == 0 || align > (1u << 20))
        return ZERO_EINVAL;
    const uint64_t N = n_ranks;
    uint64_t S = psi / N + (psi % N != 0);
    if (S % align)
        S += align - S % align;
    const uint64_t P = N * S;
    if (bucket_elems != 0 && bucket_elems < P && bucket_elems % 8 != 0)
        return ZERO_EINVAL;
    const uint64_t W = (bucket_elems == 0 || bucket_elems > P) ? P : bucket_elems;

    zero_layout_t L;
    memset(&L, 0, sizeof L);
    L.psi = psi;
    L.shard = S;
    L.psi_padded = P;
    L.pad = P - psi;
    L.bucket_elems = W;
    L.n_buckets = (P + W - 1) / W;
    L.tile_elems = ZERO_TILE_ELEMS;
    L.tiles_per_rank = zero::tiles_per_rank(S, ZERO_TILE_ELEMS);
    L.n_tiles = N * L.tiles_per_rank;
    L.n_ranks = n_ranks;
    L.stage = stage;
    L.align = align;
    const uint64_t weights = 2, grads = 2, optim = 12;  // bytes per parameter
    L.bytes_per_rank[0] = (weights + grads + optim) * psi;
    L.bytes_per_rank[1] = weights * P + grads * P + optim * S;
    L.bytes_per_rank[2] = weights * P + (grads + optim) * S;
    L.bytes_per_rank[3] = (weights + grads + optim) * S;
    const uint64_t one_collective = (N - 1) * S;
    L.comm_elems_per_rank[0] = 2 * one_collective;  // all-reduce = reduce-scatter + all-gather
    L.comm_elems_per_rank[1] = 2 * one_collective;
    L.comm_elems_per_rank[2] = 2 * one_collective;
    L.comm_elems_per_rank[3] = 3 * one_collective;  // + parameter all-gather in backward
    *out = L;
    return ZERO_OK;
}

namespace zero {

uint64_t tiles_per_rank(uint64_t S, uint64_t T)
{
    return (S + T - 1) / T + 1;  // [a, a+S) meets at most ceil(S/T) + 1 cells of the T grid
}

uint64_t tile_unit(const zero_layout_t* L, uint64_t i)
{
    const uint64_t r = i / L->shard, T = L->tile_elems;
    return r * L->tiles_per_rank + (i / T - (r * L->shard) / T);
}

}  // namespace zero

extern "C" size_t zero_workspace_bytes(const zero_layout_t* layout)
{
    if (!layout || layout->n_ranks == 0 || layout->tile_elems == 0)
        return 0;
    return (size_t)layout->n_tiles * sizeof(double);
}

/*
 * zero_segment_map -- where each model tensor's elements live among the shards.
 * "【论文解读】ZeRO" sec. 4(2): gradients are bucketed by partition and reduced at the
 * partition boundary, so a tensor that crosses a shard boundary is split between two
 * or more owners.  The tensors are laid end to end over the flat buffer in list order;
 * tensor k's piece on rank r is its intersection with [r*S, (r+1)*S).  One pass over the
 * tensors, O(n_tensors + n_ranks); the pieces come out in flat order.
 */
extern "C" int zero_segment_map(const zero_layout_t* layout, const uint64_t* tensor_elems,
                                uint64_t n_tensors, zero_segment_t* out, uint64_t capacity,
                                uint64_t* n_segments)
{
    if (!zero::layout_ok(layout) || !n_segments || (n_tensors > 0 && !tensor_elems))
        return ZERO_EINVAL;
    const uint64_t S = layout->shard;
    uint64_t total = 0, count = 0;
    for (uint64_t k = 0; k < n_tensors; ++k) {
        const uint64_t e = tensor_elems[k];
        if (e > layout->psi - total)  // also catches a sum past 2^64
            return ZERO_EINVAL;
        if (e > 0)
            count += (total + e - 1) / S - total / S + 1;
        total += e;
    }
    if (total != layout->psi)
        return ZERO_EINVAL;
    *n_segments = count;
    if (!out)
        return ZERO_OK;
    if (capacity < count)
        return ZERO_ENOMEM;
    uint64_t a = 0, w = 0;
    for (uint64_t k = 0; k < n_tensors; ++k) {
        const uint64_t b = a + tensor_elems[k];
        for (uint64_t r = a / S; a < b && r * S < b; ++r) {
            const uint64_t lo = a > r * S ? a : r * S;
            const uint64_t hi = b < (r + 1) * S ? b : (r + 1) * S;
            out[w++] = zero_segment_t{k, r, lo - a, lo - r * S, hi - lo};
        }
        a = b;
    }
    return ZERO_OK;
}

