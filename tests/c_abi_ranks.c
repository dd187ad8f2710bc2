/* The ZeRO step with its ranks spread over two processes, driven from a plain C program
 * through the rank-local entry points of libzero_shard.so; the exchanges between the two
 * are cudaMemcpy calls between their buffers (standing in for the collectives a real
 * multi-process job makes), and both "processes" run one after the other in this one
 * program, so nothing on the GPU waits on anything else.  Every output is compared bit
 * for bit with zero_step on the same layout, where all four ranks are buffers of one
 * caller.  No PyTorch, no Python.  Built and run by tests/test_c_abi.py (GPU test).
 *
 * Per step and process p (ranks 2p and 2p+1, flat [origin_p, origin_p + 2S)):
 *   1. every rank's gradient copy of p's range is copied in (the all-to-all);
 *   2. zero_reduce_shard_unscale_local over the range;
 *   3. the two processes' partial slots are exchanged, and the overflow words combined
 *      (maximum);
 *   4. zero_grad_norm;
 *   5. zero_adamw_cast_gather_local, written at origin_p of p's gathered buffer;
 *   6. the two processes' parameter ranges are exchanged (the all-gather). */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "zero.h"

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

enum { N = 4, G = 2, R = N / G, STEPS = 2 };

typedef struct proc {
    uint32_t rank_begin;
    uint64_t origin, len;
    void* recv;            /* N chunks of len bf16: rank k's copy of this range */
    float* g;              /* len */
    float* state;          /* master, m, v: len each */
    uint16_t* params;      /* psi_padded: the full gathered buffer */
    double* partials;      /* n_tiles */
    zero_step_state_t* st;
} proc_t;

int main(void)
{
    const uint64_t psi = 100003;
    zero_layout_t L;
    ZK(zero_partition(psi, N, 2, 8, 0, &L));   /* align 8: every origin a multiple of 8 */
    const uint64_t P = L.psi_padded, S = L.shard;

    /* host inputs for STEPS steps: N bf16 gradient copies per step (pads 0); master/m/v */
    uint16_t* reps = calloc((size_t)STEPS * N * P, 2);
    float* st3 = calloc(3 * P, 4);
    for (uint64_t s = 0; s < STEPS; ++s)
        for (uint64_t k = 0; k < N; ++k)
            for (uint64_t i = 0; i < psi; ++i) {
                float x = uniform((s * N + k) * 1000003ull + i, 1e-3);
                uint32_t u;
                memcpy(&u, &x, 4);
                reps[(s * N + k) * P + i] = (uint16_t)(u >> 16);
            }
    for (uint64_t i = 0; i < psi; ++i) {
        st3[i] = uniform(7ull << 40 | i, 0.02);
        st3[P + i] = uniform(8ull << 40 | i, 1e-4);
        float v = uniform(9ull << 40 | i, 1e-4);
        st3[2 * P + i] = v * v;
    }
    zero_adamw_hparams_t hp = {1e-3f, 0.9f, 0.999f, 1e-8f, 0.01f, 1e-3f, 0};  /* clip active */

    /* the one-caller step: all N ranks' buffers together */
    uint16_t* d_reps;
    float *d_g, *d_state;
    uint16_t* d_out;
    double* d_part;
    zero_step_state_t* d_st;
    CK(cudaMalloc((void**)&d_reps, (size_t)STEPS * N * P * 2));
    CK(cudaMalloc((void**)&d_g, P * 4));
    CK(cudaMalloc((void**)&d_state, 3 * P * 4));
    CK(cudaMalloc((void**)&d_out, P * 2));
    CK(cudaMalloc((void**)&d_part, zero_workspace_bytes(&L)));
    CK(cudaMalloc((void**)&d_st, sizeof(zero_step_state_t)));
    CK(cudaMemcpy(d_reps, reps, (size_t)STEPS * N * P * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_state, st3, 3 * P * 4, cudaMemcpyHostToDevice));
    CK(cudaMemset(d_out, 0, P * 2));
    ZK(zero_step_state_init(&L, 1.0f, 0, 1000, d_st, d_part, NULL));

    /* the two processes' own buffers */
    proc_t pr[G];
    for (int p = 0; p < G; ++p) {
        proc_t* q = &pr[p];
        q->rank_begin = (uint32_t)(p * R);
        q->origin = (uint64_t)p * R * S;
        q->len = (uint64_t)R * S;
        CK(cudaMalloc(&q->recv, N * q->len * 2));
        CK(cudaMalloc((void**)&q->g, q->len * 4));
        CK(cudaMalloc((void**)&q->state, 3 * q->len * 4));
        CK(cudaMalloc((void**)&q->params, P * 2));
        CK(cudaMalloc((void**)&q->partials, zero_workspace_bytes(&L)));
        CK(cudaMalloc((void**)&q->st, sizeof(zero_step_state_t)));
        for (int a = 0; a < 3; ++a)
            CK(cudaMemcpy(q->state + a * q->len, st3 + a * P + q->origin, q->len * 4,
                          cudaMemcpyHostToDevice));
        CK(cudaMemset(q->params, 0, P * 2));
        ZK(zero_step_state_init(&L, 1.0f, 0, 1000, q->st, q->partials, NULL));
    }

    const size_t ovf = offsetof(zero_step_state_t, overflow);
    const uint64_t tpr = L.tiles_per_rank;
    for (int s = 0; s < STEPS; ++s) {
        const uint16_t* step_reps = d_reps + (uint64_t)s * N * P;
        const void* rp[N];
        for (int k = 0; k < N; ++k)
            rp[k] = step_reps + (uint64_t)k * P;
        ZK(zero_step(&L, &hp, ZERO_BF16, rp, d_g, d_part, d_state, d_state + P, d_state + 2 * P,
                     d_out, d_st, NULL));

        for (int p = 0; p < G; ++p) {  /* 1 and 2 */
            proc_t* q = &pr[p];
            const void* chunk[N];
            for (int k = 0; k < N; ++k) {
                uint16_t* dst = (uint16_t*)q->recv + (uint64_t)k * q->len;
                CK(cudaMemcpy(dst, step_reps + (uint64_t)k * P + q->origin, q->len * 2,
                              cudaMemcpyDeviceToDevice));
                chunk[k] = dst;
            }
            ZK(zero_reduce_shard_unscale_local(&L, ZERO_BF16, q->rank_begin, R, chunk, q->origin,
                                               q->len, q->g, q->partials, q->st, NULL));
        }
        uint32_t flag = 0;  /* 3 */
        for (int p = 0; p < G; ++p) {
            uint32_t f;
            CK(cudaMemcpy(&f, (char*)pr[p].st + ovf, 4, cudaMemcpyDeviceToHost));
            flag = f > flag ? f : flag;
            for (int o = 0; o < G; ++o)
                if (o != p)
                    CK(cudaMemcpy(pr[o].partials + pr[p].rank_begin * tpr,
                                  pr[p].partials + pr[p].rank_begin * tpr, R * tpr * 8,
                                  cudaMemcpyDeviceToDevice));
        }
        for (int p = 0; p < G; ++p) {  /* 4 and 5 */
            proc_t* q = &pr[p];
            CK(cudaMemcpy((char*)q->st + ovf, &flag, 4, cudaMemcpyHostToDevice));
            ZK(zero_grad_norm(&L, &hp, q->partials, q->st, NULL));
            ZK(zero_adamw_cast_gather_local(&L, &hp, q->rank_begin, R, q->g, q->state,
                                            q->state + q->len, q->state + 2 * q->len,
                                            q->params + q->origin, q->st, NULL));
        }
        for (int p = 0; p < G; ++p)  /* 6 */
            for (int o = 0; o < G; ++o)
                if (o != p)
                    CK(cudaMemcpy(pr[o].params + pr[p].origin, pr[p].params + pr[p].origin,
                                  pr[p].len * 2, cudaMemcpyDeviceToDevice));
    }
    CK(cudaDeviceSynchronize());

    /* compare: state bytes, gathered parameters, g and master/m/v slices, all bit for bit */
    zero_step_state_t want;
    ZK(zero_step_state_read(d_st, &want, NULL));
    uint16_t* out = malloc(P * 2);
    float* g = malloc(P * 4);
    float* state = malloc(3 * P * 4);
    CK(cudaMemcpy(out, d_out, P * 2, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(g, d_g, P * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(state, d_state, 3 * P * 4, cudaMemcpyDeviceToHost));
    uint16_t* pout = malloc(P * 2);
    float* pbuf = malloc(3 * P * 4);
    int bad = 0;
    for (int p = 0; p < G; ++p) {
        proc_t* q = &pr[p];
        zero_step_state_t got;
        ZK(zero_step_state_read(q->st, &got, NULL));
        if (memcmp(&got, &want, sizeof got) != 0) {
            printf("process %d: step state differs\n", p);
            ++bad;
        }
        CK(cudaMemcpy(pout, q->params, P * 2, cudaMemcpyDeviceToHost));
        if (memcmp(pout, out, P * 2) != 0) {
            printf("process %d: gathered parameters differ\n", p);
            ++bad;
        }
        CK(cudaMemcpy(pbuf, q->g, q->len * 4, cudaMemcpyDeviceToHost));
        if (memcmp(pbuf, g + q->origin, q->len * 4) != 0) {
            printf("process %d: g differs\n", p);
            ++bad;
        }
        CK(cudaMemcpy(pbuf, q->state, 3 * q->len * 4, cudaMemcpyDeviceToHost));
        for (int a = 0; a < 3; ++a)
            if (memcmp(pbuf + a * q->len, state + a * P + q->origin, q->len * 4) != 0) {
                printf("process %d: optimizer state array %d differs\n", p, a);
                ++bad;
            }
    }
    printf("t %u, norm %.9g, c %.9g; two processes of two ranks each, %d mismatches\n", want.t,
           want.norm, want.clip_coef, bad);
    if (bad || want.t != STEPS || want.clip_coef >= 1.0f)
        return 1;
    printf("ok\n");
    return 0;
}
