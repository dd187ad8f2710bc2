/*
 * zsynth_host.c -- host twin of the seeded input generator (see zsynth.h).
 * Build: gcc -O2 -ffp-contract=off -fopenmp -fPIC -shared.  Threads split the index
 * range; every value depends only on (key, flat index), so the output does not depend
 * on the thread count.
 */
#include <math.h>
#include <stdint.h>

#include "zsynth.h"

uint64_t zsynth_key(uint64_t seed, uint32_t role, uint32_t step, uint32_t rank)
{
    return zs_key(seed, role, step, rank);
}

float zsynth_normal(uint64_t key, uint64_t pos) { return zs_normal(key, pos); }

float zsynth_value(int kind, uint64_t key, uint64_t i, float sigma, float scale)
{
    return zs_value(kind, key, i, sigma, scale);
}

uint16_t zsynth_f32_to_f16(float x) { return zs_f32_to_f16(x); }
uint16_t zsynth_f32_to_bf16(float x) { return zs_f32_to_bf16(x); }

static void store(void* dst, int out, uint64_t j, float x)
{
    if (out == ZS_OUT_F32)
        ((float*)dst)[j] = x;
    else if (out == ZS_OUT_BF16)
        ((uint16_t*)dst)[j] = zs_f32_to_bf16(x);
    else
        ((uint16_t*)dst)[j] = zs_f32_to_f16(x);
}

/* dst[j] = value at flat index begin + j for j < count; zero where the index >= valid_end. */
void zsynth_fill_host(void* dst, int out, int kind, uint64_t key, uint64_t begin, uint64_t count,
                      uint64_t valid_end, float sigma, float scale)
{
    int64_t n = (int64_t)count;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) {
        uint64_t i = begin + (uint64_t)j;
        float x = i < valid_end ? zs_value(kind, key, i, sigma, scale) : 0.0f;
        store(dst, out, (uint64_t)j, x);
    }
}

/* dst[j] = value at flat index idx[j] (zero where idx[j] >= valid_end). */
void zsynth_gather_host(void* dst, int out, int kind, uint64_t key, const uint64_t* idx,
                        uint64_t n, uint64_t valid_end, float sigma, float scale)
{
    int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < nn; ++j) {
        uint64_t i = idx[j];
        float x = i < valid_end ? zs_value(kind, key, i, sigma, scale) : 0.0f;
        store(dst, out, (uint64_t)j, x);
    }
}
