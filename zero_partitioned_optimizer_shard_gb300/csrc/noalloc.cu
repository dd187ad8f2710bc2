/*
 * noalloc.cu -- zero_step_static_workspace: the whole step with no caller workspace.
 *
 * Some callers cannot hand this library a scratch buffer, because they cannot allocate
 * device memory at the point where they run the optimizer: their memory manager has
 * already reserved every byte of the GPU, or they must not take the device-wide
 * synchronisation that cudaMalloc/cudaFree can cause in the middle of a training step.
 * For them this entry point keeps the step's only scratch, the per-tile sum-of-squares
 * partials, in one fixed array of static device memory declared below.  It allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *
 * The array holds ZERO_STATIC_WORKSPACE_SLOTS 8-byte slots (8 MiB).  Every GPU on which
 * this library's device code is loaded holds those 8 MiB until the process exits.
 *
 * In host code the array's name only stands for the device symbol: it is not a device
 * address.  The first call on each device looks the address up with
 * cudaGetSymbolAddress (with that device current) and caches it; the kernels get that
 * address.
 */
#include "zero_internal.h"

#include <mutex>
#include <string.h>

static __device__ __align__(256) double zero_static_partials[ZERO_STATIC_WORKSPACE_SLOTS];

namespace {

int fail_cuda(cudaError_t e)
{
    zero::record_cuda_error((int)e);  // reported by zero_last_cuda_error()
    return ZERO_ECUDA;
}

bool is_aligned16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }

/* The same invariants the other device entry points check, restated here so this
 * entry point's validation shares no code path with them (the tile grid is the
 * layout's definition, shared). */
bool layout_valid(const zero_layout_t* L)
{
    if (!L || L->n_ranks == 0 || L->n_ranks > ZERO_MAX_KERNEL_RANKS || L->psi == 0 ||
        L->shard == 0 || L->psi > (1ull << 56))
        return false;
    if (L->psi_padded != (uint64_t)L->n_ranks * L->shard || L->psi > L->psi_padded ||
        L->pad != L->psi_padded - L->psi || L->tile_elems != ZERO_TILE_ELEMS)
        return false;
    if (L->tiles_per_rank != zero::tiles_per_rank(L->shard, L->tile_elems) ||
        L->n_tiles != (uint64_t)L->n_ranks * L->tiles_per_rank)
        return false;
    const uint64_t W = L->bucket_elems;
    if (W == 0 || W > L->psi_padded || (W != L->psi_padded && W % 8 != 0))
        return false;
    return L->n_buckets == (L->psi_padded + W - 1) / W;
}

bool hp_valid(const zero_adamw_hparams_t* hp)
{
    if (!hp)
        return false;
    const float v[6] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay, hp->max_grad_norm};
    for (float x : v)
        if (!(x == x) || x > 3.0e38f || x < -3.0e38f)
            return false;
    return hp->beta1 >= 0.0f && hp->beta1 < 1.0f && hp->beta2 >= 0.0f && hp->beta2 < 1.0f &&
           hp->eps > 0.0f && hp->lr >= 0.0f &&
           (hp->params_dtype == 0 || hp->params_dtype == ZERO_BF16 || hp->params_dtype == ZERO_F16);
}

/* Device address of the static array on the current device, looked up once. */
int static_workspace(double** out)
{
    static std::mutex mu;
    static double* addr[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail_cuda(e);
    if (dev < 0 || dev >= 64)
        return ZERO_EINVAL;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, zero_static_partials);
        if (e != cudaSuccess)
            return fail_cuda(e);
        addr[dev] = (double*)p;
    }
    *out = addr[dev];
    return ZERO_OK;
}

}  // namespace

extern "C" int zero_step_static_workspace(const zero_layout_t* layout,
                                          const zero_adamw_hparams_t* hp, zero_dtype_t dtype,
                                          const void* const* replicas, float* g, float* master,
                                          float* m, float* v, uint16_t* params,
                                          zero_step_state_t* st, zero_stream_t stream)
{
    if (!layout_valid(layout) || !hp_valid(hp) || (dtype != ZERO_F16 && dtype != ZERO_BF16) ||
        !replicas || !g || !master || !m || !v || !params || !st)
        return ZERO_EINVAL;
    if (layout->n_tiles > ZERO_STATIC_WORKSPACE_SLOTS)
        return ZERO_ENOMEM;  // the problem needs more partial slots than the static array has
    const uint64_t N = layout->n_ranks, W = layout->bucket_elems, P = layout->psi_padded;
    const uint64_t nrep = layout->n_buckets * N;
    for (uint64_t i = 0; i < nrep; ++i)
        if (!replicas[i])
            return ZERO_EINVAL;
    for (uint64_t i = 0; i < nrep; ++i)
        if (!is_aligned16(replicas[i]))
            return ZERO_EALIGN;
    if (!is_aligned16(g) || !is_aligned16(master) || !is_aligned16(m) || !is_aligned16(v) ||
        !is_aligned16(params) || !is_aligned16(st))
        return ZERO_EALIGN;

    double* ws = nullptr;
    int rc = static_workspace(&ws);
    if (rc != ZERO_OK)
        return rc;
    const cudaStream_t s = (cudaStream_t)stream;

    // the array keeps whatever the previous call left: clear the slots this step adds into
    cudaError_t e = cudaMemsetAsync(ws, 0, layout->n_tiles * sizeof(double), s);
    if (e != cudaSuccess)
        return fail_cuda(e);

    for (uint64_t b = 0; b < layout->n_buckets; ++b) {
        zero::ReduceArgs a;
        memset(&a, 0, sizeof a);
        for (uint64_t k = 0; k < N; ++k)
            a.rep[k] = replicas[b * N + k];
        a.g = g;
        a.partials = ws;
        a.st = st;
        a.begin = b * W;
        a.end = a.begin + W < P ? a.begin + W : P;
        a.psi = layout->psi;
        a.shard = layout->shard;
        a.tiles_per_rank = layout->tiles_per_rank;
        a.n_ranks = layout->n_ranks;
        a.tile = layout->tile_elems;
        a.unit_first = zero::tile_unit(layout, a.begin);
        a.unit_count = zero::tile_unit(layout, a.end - 1) - a.unit_first + 1;
        e = zero::launch_reduce(a, dtype, s);
        if (e != cudaSuccess)
            return fail_cuda(e);
    }

    zero::FinalizeArgs f;
    f.partials = ws;
    f.st = st;
    f.tiles_per_rank = layout->tiles_per_rank;
    f.n_ranks = layout->n_ranks;
    f.hp = *hp;
    e = zero::launch_finalize(f, s);
    if (e != cudaSuccess)
        return fail_cuda(e);

    zero::AdamwArgs u;
    memset(&u, 0, sizeof u);
    u.g = g;
    u.master = master;
    u.m = m;
    u.v = v;
    u.out = params;
    u.st = st;
    u.err = &st->error;
    u.next_chunk = reinterpret_cast<unsigned long long*>(&st->adamw_next_chunk);
    u.done = &st->adamw_done;
    u.psi = layout->psi;
    u.psi_padded = P;
    u.beta1 = hp->beta1;
    u.beta2 = hp->beta2;
    u.eps = hp->eps;
    u.out_f16 = hp->params_dtype == ZERO_F16 ? 1u : 0u;
    e = zero::launch_adamw(u, s);
    return e == cudaSuccess ? ZERO_OK : fail_cuda(e);
}
