/*
 * zsynth.h -- seeded synthetic inputs for the ZeRO optimizer step (per-element core).
 *
 * This module generates inputs only; it holds none of the optimizer's arithmetic.  The
 * host twin (zsynth_host.c, gcc -ffp-contract=off) and the device twin (zsynth_dev.cu,
 * nvcc --fmad=false) both include this file, so every generated value is a pure function
 * of (key, flat index) and the two twins agree bit for bit: the integer hash is exact,
 * and the floating-point steps are single IEEE operations (+, *, /, sqrt), each
 * correctly rounded on both processors.
 *
 *   hash      SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom
 *             number generators", OOPSLA 2014): state advances by the golden-ratio
 *             increment 0x9e3779b97f4a7c15, output = the 64-bit mixing function below.
 *             Used counter-style: value j of stream `key` is mix64(key + j*gamma).
 *   normal    Irwin-Hall: the sum of twelve uniforms minus six.  Twelve 16-bit uniforms
 *             come from three hash outputs; their integer sum is exact, centred by
 *             12*65535/2 and scaled by 2^-16 (exact), giving mean 0, variance 1.
 *   t(3)      Student-t with 3 degrees of freedom: z0 / sqrt((z1^2 + z2^2 + z3^2) / 3).
 *   casts     float -> bfloat16 and float -> IEEE binary16, round to nearest even.
 */
#ifndef ZSYNTH_H
#define ZSYNTH_H

#include <math.h>
#include <stdint.h>

#if defined(__CUDACC__)
#define ZS_FN static __host__ __device__ __forceinline__
#else
#define ZS_FN static inline
#endif

#define ZS_GAMMA 0x9e3779b97f4a7c15ull

enum { ZS_ROLE_GRAD = 1, ZS_ROLE_MASTER = 2, ZS_ROLE_MOM = 3, ZS_ROLE_VAR = 4 };
enum { ZS_NORMAL = 0, ZS_NORMAL_SQ = 1, ZS_STUDENT_T3 = 2 };
enum { ZS_OUT_F32 = 0, ZS_OUT_BF16 = 1, ZS_OUT_F16 = 2 };

ZS_FN uint64_t zs_mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

/* One stream per (seed, role, step, rank). */
ZS_FN uint64_t zs_key(uint64_t seed, uint32_t role, uint32_t step, uint32_t rank)
{
    uint64_t a = zs_mix64(seed + ZS_GAMMA * (uint64_t)(role + 1));
    return zs_mix64(a ^ (((uint64_t)step << 32) | (uint64_t)rank));
}

ZS_FN float zs_u32_as_f32(uint32_t u)
{
    union { uint32_t u; float f; } c;
    c.u = u;
    return c.f;
}

ZS_FN uint32_t zs_f32_bits(float f)
{
    union { uint32_t u; float f; } c;
    c.f = f;
    return c.u;
}

/* Irwin-Hall(12) normal number `pos` of stream `key`. */
ZS_FN float zs_normal(uint64_t key, uint64_t pos)
{
    uint64_t base = key + 3ull * pos * ZS_GAMMA;
    int32_t s = 0;
    for (int j = 1; j <= 3; ++j) {
        uint64_t h = zs_mix64(base + (uint64_t)j * ZS_GAMMA);
        s += (int32_t)(h & 0xffff) + (int32_t)((h >> 16) & 0xffff) +
             (int32_t)((h >> 32) & 0xffff) + (int32_t)(h >> 48);
    }
    /* exact: |s - 393210| < 2^24, and the scale is a power of two */
    return (float)(s - 393210) * 0.0000152587890625f;
}

/* Student-t(3) number `i` of stream `key` (uses normals 4i .. 4i+3). */
ZS_FN float zs_student_t3(uint64_t key, uint64_t i)
{
    float z0 = zs_normal(key, 4 * i);
    float z1 = zs_normal(key, 4 * i + 1);
    float z2 = zs_normal(key, 4 * i + 2);
    float z3 = zs_normal(key, 4 * i + 3);
    float q = z1 * z1;
    q = q + z2 * z2;
    q = q + z3 * z3;
    return z0 / sqrtf(q / 3.0f);
}

/* The value at flat index i: draw * sigma, squared for ZS_NORMAL_SQ, then * scale. */
ZS_FN float zs_value(int kind, uint64_t key, uint64_t i, float sigma, float scale)
{
    float x = (kind == ZS_STUDENT_T3) ? zs_student_t3(key, i) : zs_normal(key, i);
    x = x * sigma;
    if (kind == ZS_NORMAL_SQ)
        x = x * x;
    return x * scale;
}

/* Round-to-nearest-even right shift of a 32-bit magnitude by s (1 <= s <= 31). */
ZS_FN uint32_t zs_rne_shift(uint32_t x, uint32_t s)
{
    uint32_t q = x >> s;
    uint32_t rem = x & ((1u << s) - 1u);
    uint32_t half = 1u << (s - 1);
    if (rem > half || (rem == half && (q & 1u)))
        q += 1;
    return q;
}

ZS_FN uint16_t zs_f32_to_bf16(float x)
{
    uint32_t u = zs_f32_bits(x);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)(((u >> 16) & 0x8000u) | 0x7fc0u);
    uint32_t sign = u & 0x80000000u;
    uint32_t mag = zs_rne_shift(u & 0x7fffffffu, 16);  /* carry into the exponent is correct */
    return (uint16_t)((sign >> 16) | mag);
}

ZS_FN uint16_t zs_f32_to_f16(float x)
{
    uint32_t u = zs_f32_bits(x);
    uint32_t sign = (u >> 16) & 0x8000u;
    uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u)
        return (uint16_t)(sign | 0x7e00u);           /* NaN */
    if (a >= 0x477ff000u)
        return (uint16_t)(sign | 0x7c00u);           /* >= 65520 rounds to inf */
    if (a >= 0x38800000u)                            /* >= 2^-14: normal binary16 */
        return (uint16_t)(sign | zs_rne_shift(a - 0x38000000u, 13));
    /* subnormal binary16: units of 2^-24 */
    uint32_t e = a >> 23;
    if (e < 102)
        return (uint16_t)sign;                       /* below 2^-25: rounds to zero */
    uint32_t mant = (a & 0x7fffffu) | 0x800000u;     /* value = mant * 2^(e-150) */
    return (uint16_t)(sign | zs_rne_shift(mant, 126 - e));
}

#endif /* ZSYNTH_H */
