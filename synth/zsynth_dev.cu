/*
 * zsynth_dev.cu -- device twin of the seeded input generator (see zsynth.h).
 * Build: nvcc --fmad=false (no contraction; division and sqrt stay IEEE), so each value
 * equals the host twin's bit for bit.  Input generation only: it is never on the timed
 * optimizer path.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "zsynth.h"

template <int OUT>
__global__ void k_zsynth_fill(void* __restrict__ dst, int kind, uint64_t key, uint64_t begin,
                              uint64_t count, uint64_t valid_end, float sigma, float scale)
{
    uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < count; j += stride) {
        uint64_t i = begin + j;
        float x = i < valid_end ? zs_value(kind, key, i, sigma, scale) : 0.0f;
        if (OUT == ZS_OUT_F32)
            ((float*)dst)[j] = x;
        else if (OUT == ZS_OUT_BF16)
            ((uint16_t*)dst)[j] = zs_f32_to_bf16(x);
        else
            ((uint16_t*)dst)[j] = zs_f32_to_f16(x);
    }
}

/* blocks_per_sm caps the grid (0 = 16 per SM, the whole GPU); a small cap leaves SMs for
 * kernels that run beside the generator. */
extern "C" int zsynth_fill_dev(void* dst, int out, int kind, uint64_t key, uint64_t begin,
                               uint64_t count, uint64_t valid_end, float sigma, float scale,
                               void* stream, int blocks_per_sm)
{
    if (count == 0)
        return 0;
    if (!dst || out < 0 || out > 2)
        return -1;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    uint64_t want = (count + 255) / 256;
    uint64_t cap = (uint64_t)(sms > 0 ? sms : 1) * (uint64_t)(blocks_per_sm > 0 ? blocks_per_sm : 16);
    unsigned grid = (unsigned)(want < cap ? want : cap);
    cudaStream_t s = (cudaStream_t)stream;
    if (out == ZS_OUT_F32)
        k_zsynth_fill<ZS_OUT_F32><<<grid, 256, 0, s>>>(dst, kind, key, begin, count, valid_end, sigma, scale);
    else if (out == ZS_OUT_BF16)
        k_zsynth_fill<ZS_OUT_BF16><<<grid, 256, 0, s>>>(dst, kind, key, begin, count, valid_end, sigma, scale);
    else
        k_zsynth_fill<ZS_OUT_F16><<<grid, 256, 0, s>>>(dst, kind, key, begin, count, valid_end, sigma, scale);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}
