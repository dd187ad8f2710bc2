/* One ZeRO step from a plain C program: CUDA runtime allocations and copies, the step
 * through the C ABI of libzero_shard.so, and the same step in the C oracle on the same
 * inputs, compared element by element.  No PyTorch, no Python.  Built and run by
 * tests/test_c_abi.py (GPU test).  Inputs come from a small integer hash, fixed here. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "zero.h"
#include "zero_oracle.h"

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { printf("CUDA %s line %d\n", cudaGetErrorString(e_), __LINE__); return 1; } } while (0)
#define ZK(x) do { int r_ = (x); if (r_ != ZERO_OK) { printf("zero status %d (%s) line %d\n", r_, zero_strerror(r_), __LINE__); return 1; } } while (0)

static uint32_t mix(uint64_t x)  /* SplitMix64 finaliser, top 32 bits */
{
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return (uint32_t)((x ^ (x >> 31)) >> 32);
}

static float uniform(uint64_t key, double scale)  /* in [-scale, scale) */
{
    return (float)(((double)mix(key) / 4294967296.0 * 2.0 - 1.0) * scale);
}

int main(void)
{
    const uint64_t psi = 100003, N = 4;
    zero_layout_t L;
    ZK(zero_partition(psi, (uint32_t)N, 2, 1, 0, &L));
    const uint64_t P = L.psi_padded;
    const uint64_t R = (P + 7) & ~7ull;  /* array stride: every copy and state array starts 16-byte aligned */

    /* host inputs: N bf16 gradient copies (pads 0), fp32 master / m / v */
    uint16_t* reps = calloc(N * R, 2);
    float* st3 = calloc(3 * R, 4);
    for (uint64_t k = 0; k < N; ++k)
        for (uint64_t i = 0; i < psi; ++i) {
            float x = uniform(k * 1000003ull + i, 1e-3);
            uint32_t u;
            memcpy(&u, &x, 4);
            reps[k * R + i] = (uint16_t)(u >> 16);  /* truncate to bf16 */
        }
    for (uint64_t i = 0; i < psi; ++i) {
        st3[i] = uniform(7ull << 40 | i, 0.02);
        st3[R + i] = uniform(8ull << 40 | i, 1e-4);
        float s = uniform(9ull << 40 | i, 1e-4);
        st3[2 * R + i] = s * s;
    }

    /* device buffers through the CUDA runtime */
    void* d_reps;
    float *d_g, *d_state;
    uint16_t* d_out;
    double* d_part;
    zero_step_state_t* d_st;
    CK(cudaMalloc(&d_reps, N * R * 2));
    CK(cudaMalloc((void**)&d_g, P * 4));
    CK(cudaMalloc((void**)&d_state, 3 * R * 4));
    CK(cudaMalloc((void**)&d_out, P * 2));
    CK(cudaMalloc((void**)&d_part, zero_workspace_bytes(&L)));
    CK(cudaMalloc((void**)&d_st, sizeof(zero_step_state_t)));
    CK(cudaMemcpy(d_reps, reps, N * R * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_state, st3, 3 * R * 4, cudaMemcpyHostToDevice));
    const void* rp[4];
    for (uint64_t k = 0; k < N; ++k)
        rp[k] = (const char*)d_reps + k * R * 2;
    zero_adamw_hparams_t hp = {1e-3f, 0.9f, 0.999f, 1e-8f, 0.01f, 1.0f, 0};
    ZK(zero_step_state_init(&L, 1.0f, 0, 1000, d_st, d_part, NULL));
    for (int step = 0; step < 2; ++step)
        ZK(zero_step(&L, &hp, ZERO_BF16, rp, d_g, d_part, d_state, d_state + R, d_state + 2 * R,
                     d_out, d_st, NULL));
    zero_step_state_t s;
    ZK(zero_step_state_read(d_st, &s, NULL));
    float* g = malloc(P * 4);
    float* state = malloc(3 * R * 4);
    uint16_t* out = malloc(P * 2);
    CK(cudaMemcpy(g, d_g, P * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(state, d_state, 3 * R * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out, d_out, P * 2, cudaMemcpyDeviceToHost));

    /* the oracle, two steps on the same inputs */
    oracle_layout_t ol;
    if (oracle_partition(psi, N, 2, 1, 0, &ol) != 0)
        return 1;
    oracle_hparams_t ohp = {1e-3f, 0.9f, 0.999f, 1e-8f, 0.01f, 1.0f, 0};
    oracle_scaler_t sc = {1.0f, 0, 1000, 0, 0, 0};
    oracle_report_t rep;
    const uint16_t* orp[4];
    for (uint64_t k = 0; k < N; ++k)
        orp[k] = reps + k * R;
    float* og = calloc(P, 4);
    uint16_t* oout = calloc(P, 2);
    for (int step = 0; step < 2; ++step)
        if (oracle_step(&ol, &ohp, ORACLE_BF16, orp, og, st3, st3 + R, st3 + 2 * R, oout, &sc, &rep) != 0)
            return 1;

    if (s.t != rep.t || s.skip != rep.skipped || fabs(s.norm - rep.norm) > 1e-5 * rep.norm) {
        printf("scalars differ: t %u/%u norm %.17g/%.17g\n", s.t, rep.t, s.norm, rep.norm);
        return 1;
    }
    uint64_t exact = 0, bad = 0;
    for (uint64_t i = 0; i < P; ++i) {
        if (memcmp(&g[i], &og[i], 4) != 0)
            ++bad;
        for (int a = 0; a < 3; ++a) {
            const float x = state[a * R + i], y = st3[a * R + i];
            if (memcmp(&x, &y, 4) == 0)
                ++exact;
            else if (!(fabs((double)x - y) <= 1e-5 * fabs((double)y) + 1e-30))
                ++bad;
        }
        const int d = (int)out[i] - (int)oout[i];
        if (d > 1 || d < -1)
            ++bad;
    }
    printf("norm %.9g (oracle %.9g), c %.9g, t %u; state elements exact %llu of %llu; bad %llu\n",
           s.norm, rep.norm, s.clip_coef, s.t, (unsigned long long)exact,
           (unsigned long long)(3 * P), (unsigned long long)bad);
    if (bad)
        return 1;
    printf("ok\n");
    return 0;
}
