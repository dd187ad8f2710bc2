/*
 * api.cu -- the C entry points of include/zero.h: argument checks, then kernel launches.
 *
 * Every check runs on the host before anything is enqueued, so a rejected call leaves
 * all buffers and the stream untouched.  No entry point allocates device memory.
 */
#include "zero_internal.h"

#include <atomic>
#include <mutex>
#include <stddef.h>
#include <string.h>

namespace zero {

/* The invariants zero_partition establishes; the kernels' indexing relies on them. */
bool layout_ok(const zero_layout_t* L)
{
    if (!L || L->n_ranks == 0 || L->n_ranks > ZERO_MAX_RANKS || L->psi == 0 || L->shard == 0)
        return false;
    if (L->psi_padded / L->n_ranks != L->shard || L->psi_padded % L->n_ranks != 0)
        return false;
    if (L->psi > L->psi_padded || L->pad != L->psi_padded - L->psi || L->psi > (1ull << 56))
        return false;
    if (L->tile_elems != ZERO_TILE_ELEMS)
        return false;
    if (L->tiles_per_rank != tiles_per_rank(L->shard, L->tile_elems) ||
        L->n_tiles != (uint64_t)L->n_ranks * L->tiles_per_rank)
        return false;
    const uint64_t W = L->bucket_elems;
    if (W == 0 || W > L->psi_padded || (W != L->psi_padded && W % 8 != 0))
        return false;
    return L->n_buckets == (L->psi_padded + W - 1) / W;
}

namespace {
thread_local int g_last_cuda_error = 0;

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess)
        return ZERO_OK;
    g_last_cuda_error = (int)e;
    return ZERO_ECUDA;
}

bool aligned16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }

bool kernel_layout_ok(const zero_layout_t* L)
{
    return layout_ok(L) && L->n_ranks <= ZERO_MAX_KERNEL_RANKS;
}

bool hparams_ok(const zero_adamw_hparams_t* hp)
{
    if (!hp)
        return false;
    const float vals[6] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay, hp->max_grad_norm};
    for (float x : vals)
        if (!(x == x) || x > 3.0e38f || x < -3.0e38f)
            return false;
    return hp->beta1 >= 0.0f && hp->beta1 < 1.0f && hp->beta2 >= 0.0f && hp->beta2 < 1.0f &&
           hp->eps > 0.0f && hp->lr >= 0.0f &&
           (hp->params_dtype == 0 || hp->params_dtype == ZERO_BF16 || hp->params_dtype == ZERO_F16);
}

int reduce_window(const zero_layout_t* L, zero_dtype_t dtype, const void* const* replicas,
                  uint64_t begin, uint64_t count, float* g, double* partials,
                  zero_step_state_t* st, cudaStream_t stream)
{
    ReduceArgs a;
    memset(&a, 0, sizeof a);
    for (uint32_t k = 0; k < L->n_ranks; ++k)
        a.rep[k] = replicas[k];
    a.g = g;
    a.partials = partials;
    a.st = st;
    a.begin = begin;
    a.end = begin + count;
    a.psi = L->psi;
    a.shard = L->shard;
    a.tiles_per_rank = L->tiles_per_rank;
    a.n_ranks = L->n_ranks;
    a.tile = L->tile_elems;
    a.unit_first = tile_unit(L, begin);
    a.unit_count = tile_unit(L, a.end - 1) - a.unit_first + 1;
    return cuda_status(launch_reduce(a, dtype, stream));
}

int check_reduce_args(const zero_layout_t* L, zero_dtype_t dtype, const void* const* replicas,
                      uint64_t begin, uint64_t count, const float* g, const double* partials,
                      const zero_step_state_t* st, bool need_g = true)
{
    if (!kernel_layout_ok(L) || (dtype != ZERO_F16 && dtype != ZERO_BF16) || !replicas)
        return ZERO_EINVAL;
    if (count == 0 || begin >= L->psi_padded || count > L->psi_padded - begin)
        return ZERO_EINVAL;
    if ((need_g && !g) || !partials || !st)
        return ZERO_EINVAL;
    for (uint32_t k = 0; k < L->n_ranks; ++k)
        if (!replicas[k])
            return ZERO_EINVAL;
    if (begin % 8 != 0 || (need_g && !aligned16(g)) || !aligned16(partials) || !aligned16(st))
        return ZERO_EALIGN;
    for (uint32_t k = 0; k < L->n_ranks; ++k)
        if (!aligned16(replicas[k]))
            return ZERO_EALIGN;
    return ZERO_OK;
}

int check_adamw_args(const zero_layout_t* L, const zero_adamw_hparams_t* hp, const float* g,
                     const float* master, const float* m, const float* v, const uint16_t* params,
                     const zero_step_state_t* st, bool need_g = true)
{
    if (!kernel_layout_ok(L) || !hparams_ok(hp) || (need_g && !g) || !master || !m || !v ||
        !params || !st)
        return ZERO_EINVAL;
    if ((need_g && !aligned16(g)) || !aligned16(master) || !aligned16(m) || !aligned16(v) ||
        !aligned16(params) || !aligned16(st))
        return ZERO_EALIGN;
    return ZERO_OK;
}

int grad_norm(const zero_layout_t* L, const zero_adamw_hparams_t* hp, double* partials,
              zero_step_state_t* st, cudaStream_t stream)
{
    FinalizeArgs a;
    a.partials = partials;
    a.st = st;
    a.tiles_per_rank = L->tiles_per_rank;
    a.n_ranks = L->n_ranks;
    a.hp = *hp;
    return cuda_status(launch_finalize(a, stream));
}

int adamw(const zero_layout_t* L, const zero_adamw_hparams_t* hp, const float* g, float* master,
          float* m, float* v, uint16_t* params, const zero_step_state_t* st, cudaStream_t stream,
          bool host_state = false)
{
    AdamwArgs a;
    memset(&a, 0, sizeof a);
    a.g = g;
    a.master = master;
    a.m = m;
    a.v = v;
    a.out = params;
    a.st = st;
    a.err = const_cast<uint32_t*>(&st->error);
    a.next_chunk = reinterpret_cast<unsigned long long*>(const_cast<uint64_t*>(&st->adamw_next_chunk));
    a.done = const_cast<uint32_t*>(&st->adamw_done);
    a.psi = L->psi;
    a.psi_padded = L->psi_padded;
    a.beta1 = hp->beta1;
    a.beta2 = hp->beta2;
    a.eps = hp->eps;
    a.out_f16 = hp->params_dtype == ZERO_F16 ? 1u : 0u;
    return cuda_status(host_state ? launch_adamw_host_state(a, stream) : launch_adamw(a, stream));
}

/* AdamW for the re-reading schedule: g formed again from the two gradient copies. */
int adamw_rereduce(const zero_layout_t* L, const zero_adamw_hparams_t* hp, zero_dtype_t dtype,
                   const void* rep0, const void* rep1, float* master, float* m, float* v,
                   uint16_t* params, const zero_step_state_t* st, cudaStream_t stream)
{
    AdamwArgs a;
    memset(&a, 0, sizeof a);
    a.master = master;
    a.m = m;
    a.v = v;
    a.out = params;
    a.st = st;
    a.err = const_cast<uint32_t*>(&st->error);
    a.next_chunk = reinterpret_cast<unsigned long long*>(const_cast<uint64_t*>(&st->adamw_next_chunk));
    a.done = const_cast<uint32_t*>(&st->adamw_done);
    a.psi = L->psi;
    a.psi_padded = L->psi_padded;
    a.beta1 = hp->beta1;
    a.beta2 = hp->beta2;
    a.eps = hp->eps;
    a.out_f16 = hp->params_dtype == ZERO_F16 ? 1u : 0u;
    a.rep0 = static_cast<const uint16_t*>(rep0);
    a.rep1 = static_cast<const uint16_t*>(rep1);
    a.grad_f16 = dtype == ZERO_F16 ? 1u : 0u;
    return cuda_status(launch_adamw_rereduce(a, stream));
}

/* The whole step as ONE cooperative launch when the layout takes it (fused.cu: same bits
 * as the three launches).  *done tells whether it was enqueued; it is not when the layout
 * takes the three launches, or when the cooperative launch is refused because fewer
 * blocks fit on the GPU than the occupancy query promised (another context holds part of
 * it): then nothing was enqueued.  replicas: the N copies, each from flat 0. */
int fused_step(const zero_layout_t* L, const zero_adamw_hparams_t* hp, zero_dtype_t dtype,
               const void* const* replicas, float* g, double* partials, float* master, float* m,
               float* v, uint16_t* params, zero_step_state_t* st, cudaStream_t s, bool* done)
{
    *done = false;
    const int shape = fused_shape(L, dtype);
    if (shape <= 0)
        return ZERO_OK;
    FusedArgs f;
    memset(&f, 0, sizeof f);
    for (uint64_t k = 0; k < L->n_ranks; ++k)
        f.rep[k] = replicas[k];
    f.g = g;
    f.partials = partials;
    f.master = master;
    f.m = m;
    f.v = v;
    f.out = params;
    f.st = st;
    f.psi = L->psi;
    f.psi_padded = L->psi_padded;
    f.shard = L->shard;
    f.tiles_per_rank = L->tiles_per_rank;
    f.n_ranks = L->n_ranks;
    f.out_f16 = hp->params_dtype == ZERO_F16 ? 1u : 0u;
    f.hp = *hp;
    const cudaError_t e = launch_step_fused(f, dtype, L->n_tiles, shape, s);
    if (e == cudaErrorCooperativeLaunchTooLarge) {
        cudaGetLastError();  // nothing was enqueued: the caller takes the three launches
        return ZERO_OK;
    }
    *done = e == cudaSuccess;
    return cuda_status(e);
}

/* The device address of `bytes` of page-locked host memory at p (cudaHostAlloc or
 * cudaHostRegister, which UVA maps into the device's address space), or null when any
 * part of it is not such memory: pageable, device or unknown pointers are refused. */
void* pinned_host_device_ptr(const void* p, uint64_t bytes)
{
    const char* ends[2] = {static_cast<const char*>(p), static_cast<const char*>(p) + bytes - 1};
    void* dev[2] = {nullptr, nullptr};
    for (int k = 0; k < 2; ++k) {
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, ends[k]) != cudaSuccess) {
            cudaGetLastError();  // clear the (non-sticky) error the query left
            return nullptr;
        }
        if (at.type != cudaMemoryTypeHost || !at.devicePointer)
            return nullptr;
        dev[k] = at.devicePointer;
    }
    // one mapping: the last byte's device address lies exactly bytes-1 past the first's
    if (static_cast<char*>(dev[1]) - static_cast<char*>(dev[0]) != (ptrdiff_t)(bytes - 1))
        return nullptr;
    return dev[0];
}

}  // namespace

void record_cuda_error(int e) { g_last_cuda_error = e; }

int sm_count()
{
    static std::mutex mu;
    static int count[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    if (count[dev & 63] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        count[dev & 63] = n > 0 ? n : 1;
    }
    return count[dev & 63];
}

bool adamw_evict_first(uint64_t n, uint64_t bytes_per_elem)
{
    static std::atomic<long long> l2[64];  // per device; a race only repeats the query
    int dev = 0;
    cudaGetDevice(&dev);
    long long bytes = l2[dev & 63].load(std::memory_order_relaxed);
    if (bytes == 0) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev);
        bytes = v > 0 ? v : 1;
        l2[dev & 63].store(bytes, std::memory_order_relaxed);
    }
    return n * bytes_per_elem >= 16ull * (uint64_t)bytes;
}

}  // namespace zero

using namespace zero;

extern "C" int zero_step_state_init(const zero_layout_t* layout, float loss_scale, uint32_t dynamic,
                                    uint32_t growth_interval, zero_step_state_t* st,
                                    double* partials, zero_stream_t stream)
{
    const NvtxRange range("zero_step_state_init");
    if (!kernel_layout_ok(layout) || !st || !partials || !(loss_scale > 0.0f) || loss_scale > 3.0e38f)
        return ZERO_EINVAL;
    if (!aligned16(st) || !aligned16(partials))
        return ZERO_EALIGN;
    InitArgs a;
    a.st = st;
    a.partials = partials;
    a.n_tiles = layout->n_tiles;
    a.loss_scale = loss_scale;
    a.dynamic = dynamic ? 1u : 0u;
    a.growth_interval = growth_interval;
    a.n_ranks = layout->n_ranks;
    return cuda_status(launch_state_init(a, (cudaStream_t)stream));
}

extern "C" int zero_step_state_read(const zero_step_state_t* st, zero_step_state_t* host_out,
                                    zero_stream_t stream)
{
    if (!st || !host_out)
        return ZERO_EINVAL;
    cudaError_t e = cudaMemcpyAsync(host_out, st, sizeof *st, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize((cudaStream_t)stream);
    return cuda_status(e);
}

extern "C" int zero_step_state_write(zero_step_state_t* st, const zero_step_state_t* host_in,
                                     zero_stream_t stream)
{
    if (!st || !host_in)
        return ZERO_EINVAL;
    if (!aligned16(st))
        return ZERO_EALIGN;
    // the kernels' internal counters start every step at 0, whatever the copy holds (a
    // stale chunk counter would make the AdamW pass skip chunks)
    zero_step_state_t s = *host_in;
    s.arrivals = 0;
    s.launch_arrivals = 0;
    s.adamw_next_chunk = 0;
    s.adamw_done = 0;
    cudaError_t e = cudaMemcpyAsync(st, &s, sizeof s, cudaMemcpyHostToDevice, (cudaStream_t)stream);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize((cudaStream_t)stream);  // s lives until the copy is done
    return cuda_status(e);
}

extern "C" int zero_reduce_shard_unscale(const zero_layout_t* layout, zero_dtype_t dtype,
                                         const void* const* replicas, uint64_t begin, uint64_t count,
                                         float* g, double* partials, zero_step_state_t* st,
                                         zero_stream_t stream)
{
    const NvtxRange range("zero_reduce_shard_unscale");
    const int rc = check_reduce_args(layout, dtype, replicas, begin, count, g, partials, st);
    if (rc != ZERO_OK)
        return rc;
    return reduce_window(layout, dtype, replicas, begin, count, g, partials, st, (cudaStream_t)stream);
}

extern "C" int zero_grad_norm(const zero_layout_t* layout, const zero_adamw_hparams_t* hp,
                              double* partials, zero_step_state_t* st, zero_stream_t stream)
{
    const NvtxRange range("zero_grad_norm");
    if (!kernel_layout_ok(layout) || !hparams_ok(hp) || !partials || !st)
        return ZERO_EINVAL;
    if (!aligned16(partials) || !aligned16(st))
        return ZERO_EALIGN;
    return grad_norm(layout, hp, partials, st, (cudaStream_t)stream);
}

extern "C" int zero_adamw_cast_gather(const zero_layout_t* layout, const zero_adamw_hparams_t* hp,
                                      const float* g, float* master, float* m, float* v,
                                      uint16_t* params, const zero_step_state_t* st,
                                      zero_stream_t stream)
{
    const NvtxRange range("zero_adamw_cast_gather");
    const int rc = check_adamw_args(layout, hp, g, master, m, v, params, st);
    if (rc != ZERO_OK)
        return rc;
    return adamw(layout, hp, g, master, m, v, params, st, (cudaStream_t)stream);
}

extern "C" int zero_adamw_cast_gather_host_state(const zero_layout_t* layout,
                                                 const zero_adamw_hparams_t* hp, const float* g,
                                                 float* master, float* m, float* v,
                                                 uint16_t* params, const zero_step_state_t* st,
                                                 zero_stream_t stream)
{
    const NvtxRange range("zero_adamw_cast_gather_host_state");
    const int rc = check_adamw_args(layout, hp, g, master, m, v, params, st);
    if (rc != ZERO_OK)
        return rc;
    const uint64_t bytes = layout->psi_padded * sizeof(float);
    float* dm[3] = {master, m, v};
    for (float*& x : dm) {
        x = static_cast<float*>(pinned_host_device_ptr(x, bytes));
        if (!x)
            return ZERO_EINVAL;
    }
    return adamw(layout, hp, g, dm[0], dm[1], dm[2], params, st, (cudaStream_t)stream, true);
}

/* Ranks [rank_begin, rank_begin + rank_count) held by one process: their flat range
 * starts at origin = rank_begin*S and is local_len = rank_count*S long.  ZERO_EALIGN when
 * origin is not a multiple of 8 (partition with align = 8 for rank-local buffers). */
namespace zero {
namespace {
int local_range(const zero_layout_t* L, uint32_t rank_begin, uint32_t rank_count,
                uint64_t& origin, uint64_t& local_len)
{
    if (rank_count == 0 || rank_begin >= L->n_ranks || rank_count > L->n_ranks - rank_begin)
        return ZERO_EINVAL;
    origin = (uint64_t)rank_begin * L->shard;
    local_len = (uint64_t)rank_count * L->shard;
    return origin % 8 == 0 ? ZERO_OK : ZERO_EALIGN;
}
}  // namespace
}  // namespace zero

extern "C" int zero_reduce_shard_unscale_local(const zero_layout_t* layout, zero_dtype_t dtype,
                                               uint32_t rank_begin, uint32_t rank_count,
                                               const void* const* replicas, uint64_t begin,
                                               uint64_t count, float* g_local, double* partials,
                                               zero_step_state_t* st, zero_stream_t stream)
{
    const NvtxRange range("zero_reduce_shard_unscale_local");
    if (!kernel_layout_ok(layout))
        return ZERO_EINVAL;
    uint64_t origin = 0, len = 0;
    int rc = local_range(layout, rank_begin, rank_count, origin, len);
    if (rc == ZERO_EINVAL)
        return rc;
    if (count == 0 || begin < origin || begin >= origin + len || count > origin + len - begin)
        return ZERO_EINVAL;
    const int rc_args = check_reduce_args(layout, dtype, replicas, begin, count, g_local, partials, st);
    if (rc_args != ZERO_OK)
        return rc_args;
    if (rc != ZERO_OK)
        return rc;
    // the kernel indexes g by the flat index: hand it the address flat 0 would have, an
    // integer offset that it never dereferences below origin (the window starts there)
    float* g_flat = reinterpret_cast<float*>(reinterpret_cast<uintptr_t>(g_local) - origin * sizeof(float));
    return reduce_window(layout, dtype, replicas, begin, count, g_flat, partials, st,
                         (cudaStream_t)stream);
}

extern "C" int zero_adamw_cast_gather_local(const zero_layout_t* layout,
                                            const zero_adamw_hparams_t* hp, uint32_t rank_begin,
                                            uint32_t rank_count, const float* g_local,
                                            float* master_local, float* m_local, float* v_local,
                                            uint16_t* params_local, const zero_step_state_t* st,
                                            zero_stream_t stream)
{
    const NvtxRange range("zero_adamw_cast_gather_local");
    if (!kernel_layout_ok(layout))
        return ZERO_EINVAL;
    uint64_t origin = 0, len = 0;
    int rc = local_range(layout, rank_begin, rank_count, origin, len);
    if (rc == ZERO_EINVAL)
        return rc;
    const int rc_args = check_adamw_args(layout, hp, g_local, master_local, m_local, v_local,
                                         params_local, st);
    if (rc_args != ZERO_OK)
        return rc_args;
    if (rc != ZERO_OK)
        return rc;
    // the same pass over the local range: its first psi - origin elements (if any) are
    // parameters, the rest padding
    zero_layout_t local = *layout;
    local.psi = layout->psi > origin ? (layout->psi - origin < len ? layout->psi - origin : len) : 0;
    local.psi_padded = len;
    return adamw(&local, hp, g_local, master_local, m_local, v_local, params_local, st,
                 (cudaStream_t)stream);
}

extern "C" int zero_step(const zero_layout_t* layout, const zero_adamw_hparams_t* hp,
                         zero_dtype_t dtype, const void* const* replicas, float* g, double* partials,
                         float* master, float* m, float* v, uint16_t* params, zero_step_state_t* st,
                         zero_stream_t stream)
{
    const NvtxRange range("zero_step");
    if (!kernel_layout_ok(layout) || !replicas)
        return ZERO_EINVAL;
    // g == NULL: the re-reading schedule (N = 2, one window over resident copies)
    const bool reread = g == nullptr;
    if (reread && (layout->n_ranks != 2 || layout->n_buckets != 1))
        return ZERO_EINVAL;
    const uint64_t W = layout->bucket_elems, P = layout->psi_padded, N = layout->n_ranks;
    for (uint64_t b = 0; b < layout->n_buckets; ++b) {
        const uint64_t begin = b * W, count = begin + W < P ? W : P - begin;
        int rc = check_reduce_args(layout, dtype, replicas + b * N, begin, count, g, partials, st,
                                   !reread);
        if (rc != ZERO_OK)
            return rc;
    }
    int rc = check_adamw_args(layout, hp, g, master, m, v, params, st, !reread);
    if (rc != ZERO_OK)
        return rc;
    if (!aligned16(partials))
        return ZERO_EALIGN;
    const cudaStream_t s = (cudaStream_t)stream;
    bool done = false;
    rc = fused_step(layout, hp, dtype, replicas, g, partials, master, m, v, params, st, s, &done);
    if (done || rc != ZERO_OK)
        return rc;
    for (uint64_t b = 0; b < layout->n_buckets; ++b) {
        const uint64_t begin = b * W, count = begin + W < P ? W : P - begin;
        rc = reduce_window(layout, dtype, replicas + b * N, begin, count, g, partials, st, s);
        if (rc != ZERO_OK)
            return rc;
    }
    rc = grad_norm(layout, hp, partials, st, s);
    if (rc != ZERO_OK)
        return rc;
    if (reread)
        return adamw_rereduce(layout, hp, dtype, replicas[0], replicas[1], master, m, v, params,
                              st, s);
    return adamw(layout, hp, g, master, m, v, params, st, s);
}

extern "C" int zero_step_launches(const zero_layout_t* layout, zero_dtype_t dtype)
{
    if (!kernel_layout_ok(layout) || (dtype != ZERO_F16 && dtype != ZERO_BF16))
        return ZERO_EINVAL;
    return fused_shape(layout, dtype) > 0 ? 1 : (int)(layout->n_buckets + 2);
}

extern "C" int zero_step_host(const zero_layout_t* layout, const zero_adamw_hparams_t* hp,
                              zero_dtype_t dtype, const void* const* host_replicas, void* staging,
                              uint64_t staging_bytes, float* g, double* partials, float* master,
                              float* m, float* v, uint16_t* params, zero_step_state_t* st,
                              zero_step_state_t* host_state_out, zero_stream_t stream,
                              zero_stream_t copy_stream)
{
    const NvtxRange range("zero_step_host");
    if (!kernel_layout_ok(layout) || (dtype != ZERO_F16 && dtype != ZERO_BF16) || !host_replicas ||
        !staging || stream == copy_stream)
        return ZERO_EINVAL;
    const uint64_t W = layout->bucket_elems, P = layout->psi_padded, N = layout->n_ranks;
    for (uint64_t k = 0; k < N; ++k)
        if (!host_replicas[k])
            return ZERO_EINVAL;
    if (!aligned16(staging) || (W % 8 != 0 && layout->n_buckets > 1))
        return ZERO_EALIGN;
    const uint64_t slot_elems = (W + 7) / 8 * 8;  // keeps every staged copy 16-byte aligned
    if (staging_bytes / 2 / N / 2 < slot_elems)
        return ZERO_ENOMEM;
    int rc = check_adamw_args(layout, hp, g, master, m, v, params, st);
    if (rc != ZERO_OK)
        return rc;
    if (!partials)
        return ZERO_EINVAL;
    if (!aligned16(partials))
        return ZERO_EALIGN;

    const cudaStream_t s = (cudaStream_t)stream, cs = (cudaStream_t)copy_stream;
    // a small layout in one bucket whose copies all lie in page-locked host memory: the
    // single launch reads them where they are, over the CPU-GPU link (its replica reads are
    // plain global loads), so the transfer overlaps the sums instead of preceding the
    // launch, and nothing is staged
    if (layout->n_buckets == 1 && fused_shape(layout, dtype) > 0) {
        const void* direct[ZERO_MAX_KERNEL_RANKS];
        bool mapped = true;
        for (uint64_t k = 0; k < N && mapped; ++k) {
            direct[k] = pinned_host_device_ptr(host_replicas[k], P * 2);
            mapped = aligned16(direct[k]);
        }
        bool fused = false;
        if (mapped)
            rc = fused_step(layout, hp, dtype, direct, g, partials, master, m, v, params, st, s, &fused);
        if (rc != ZERO_OK)
            return rc;
        if (fused)
            return host_state_out ? cuda_status(cudaMemcpyAsync(host_state_out, st, sizeof *st,
                                                                cudaMemcpyDeviceToHost, s))
                                  : ZERO_OK;
        // not mapped, or the cooperative launch was refused: stage the copies
    }
    cudaEvent_t start, filled[2], consumed[2];
    cudaError_t e = cudaEventCreateWithFlags(&start, cudaEventDisableTiming);
    int made = e == cudaSuccess ? 1 : 0;
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
        e = cudaEventCreateWithFlags(&filled[i], cudaEventDisableTiming);
        made += e == cudaSuccess;
        if (e == cudaSuccess) {
            e = cudaEventCreateWithFlags(&consumed[i], cudaEventDisableTiming);
            made += e == cudaSuccess;
        }
    }
    // the staging ring may still be read by earlier work on `stream`
    if (e == cudaSuccess)
        e = cudaEventRecord(start, s);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(cs, start, 0);
    uint16_t* ring = (uint16_t*)staging;
    const void* reps[ZERO_MAX_KERNEL_RANKS];
    bool fused = false;
    for (uint64_t b = 0; b < layout->n_buckets && e == cudaSuccess && rc == ZERO_OK; ++b) {
        const int slot = (int)(b & 1);
        const uint64_t begin = b * W, count = begin + W < P ? W : P - begin;
        if (b >= 2)
            e = cudaStreamWaitEvent(cs, consumed[slot], 0);
        for (uint64_t k = 0; k < N && e == cudaSuccess; ++k) {
            uint16_t* dst = ring + ((uint64_t)slot * N + k) * slot_elems;
            const uint16_t* src = (const uint16_t*)host_replicas[k] + begin;
            e = cudaMemcpyAsync(dst, src, count * 2, cudaMemcpyHostToDevice, cs);
            reps[k] = dst;
        }
        if (e == cudaSuccess)
            e = cudaEventRecord(filled[slot], cs);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(s, filled[slot], 0);
        // one bucket of a small layout: the whole step as one launch, once it has arrived
        if (e == cudaSuccess && layout->n_buckets == 1)
            rc = fused_step(layout, hp, dtype, reps, g, partials, master, m, v, params, st, s,
                            &fused);
        if (e == cudaSuccess && rc == ZERO_OK && !fused)
            rc = reduce_window(layout, dtype, reps, begin, count, g, partials, st, s);
        if (e == cudaSuccess && rc == ZERO_OK)
            e = cudaEventRecord(consumed[slot], s);
    }
    if (e == cudaSuccess && rc == ZERO_OK && !fused)
        rc = grad_norm(layout, hp, partials, st, s);
    if (e == cudaSuccess && rc == ZERO_OK && !fused)
        rc = adamw(layout, hp, g, master, m, v, params, st, s);
    if (e == cudaSuccess && rc == ZERO_OK && host_state_out)
        e = cudaMemcpyAsync(host_state_out, st, sizeof *st, cudaMemcpyDeviceToHost, s);
    // destroying a recorded event is allowed; its resources go when the work completes
    if (made >= 1)
        cudaEventDestroy(start);
    for (int i = 0; i < 2; ++i) {
        if (made >= 2 + 2 * i)
            cudaEventDestroy(filled[i]);
        if (made >= 3 + 2 * i)
            cudaEventDestroy(consumed[i]);
    }
    if (e != cudaSuccess)
        return cuda_status(e);
    return rc;
}

extern "C" const char* zero_strerror(int status)
{
    switch (status) {
    case ZERO_OK: return "ok";
    case ZERO_EINVAL: return "invalid argument";
    case ZERO_EALIGN: return "pointer or window not aligned (16-byte pointers, window start a multiple of 8)";
    case ZERO_ENOMEM: return "caller-provided buffer too small";
    case ZERO_ECUDA: return "CUDA launch or copy failed";
    case ZERO_ETIMEOUT: return "bounded device wait timed out";
    default: return "unknown status";
    }
}

extern "C" int zero_last_cuda_error(void) { return g_last_cuda_error; }
