/* A plain C99 caller of the whole block, as an application without Python
 * would use it: a plan, device buffers from cudaMalloc, weight packing, a
 * prompt with a KV cache and one decode step on one stream, then a check
 * that the prompt's rows and the decoded token equal the rows of the same
 * 65 tokens run as one prompt without a cache (normwise error <= 2e-2, the
 * bf16 bound).
 * Prints "ok" and exits 0 on success.  Shapes: d_model 512, 8 heads of 64,
 * SwiGLU d_ffn 1536, 2 logical shards, bf16. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "tp.h"

#define D 512
#define NH 8
#define DH (D / NH)
#define FF 1536
#define TP 2
#define T 64          /* prompt tokens */
#define CAP (T + 1)   /* cache positions: the prompt and one decoded token */

#define TP_CHECK(call)                                                                  \
    do {                                                                                \
        tp_status s_ = (call);                                                          \
        if (s_ != TP_OK) {                                                              \
            fprintf(stderr, "%s:%d: %s -> %s %s\n", __FILE__, __LINE__, #call,          \
                    tp_status_string(s_), tp_last_cuda_error());                        \
            return 1;                                                                   \
        }                                                                               \
    } while (0)
#define CU_CHECK(call)                                                                  \
    do {                                                                                \
        cudaError_t e_ = (call);                                                        \
        if (e_ != cudaSuccess) {                                                        \
            fprintf(stderr, "%s:%d: %s -> %s\n", __FILE__, __LINE__, #call,             \
                    cudaGetErrorString(e_));                                            \
            return 1;                                                                   \
        }                                                                               \
    } while (0)

/* fp32 -> bf16 bits, round to nearest even (finite inputs) */
static uint16_t to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* uniform in [-a, a) from a 64-bit linear congruential generator */
static float uniform(uint64_t* state, float a) {
    *state = *state * 6364136223846793005ull + 1442695040888963407ull;
    return a * ((float)(*state >> 40) / 8388608.0f - 1.0f);
}

/* a device copy of n bf16 values drawn uniform in [-a, a) */
static void* device_bf16(size_t n, float a, uint64_t* state) {
    uint16_t* h = (uint16_t*)malloc(n * sizeof(uint16_t));
    void* d = NULL;
    size_t i;
    if (!h) return NULL;
    for (i = 0; i < n; ++i) h[i] = to_bf16(uniform(state, a));
    if (cudaMalloc(&d, n * sizeof(uint16_t)) != cudaSuccess ||
        cudaMemcpy(d, h, n * sizeof(uint16_t), cudaMemcpyHostToDevice) != cudaSuccess)
        d = NULL;
    free(h);
    return d;
}

int main(void) {
    tp_plan_t plan = NULL;
    size_t packed_bytes = 0, ws_bytes = 0, ws1 = 0, i;
    uint64_t rng = 42;
    void *w[7], *packed = NULL, *ws = NULL, *x = NULL, *kc = NULL, *vc = NULL;
    float *y_all = NULL, *y_prompt = NULL, *y_tok = NULL;
    const size_t rows[7] = {D, D, D, D, FF, FF, D}, cols[7] = {D, D, D, D, D, D, FF};
    const size_t cache_bytes = (size_t)NH * CAP * DH * sizeof(uint16_t);
    static float h_all[CAP * D], h_prompt[T * D], h_tok[D];
    double num = 0.0, den = 0.0;
    int k;

    TP_CHECK(tp_plan_create_ex(D, NH, FF, TP, TP_ACT_SWIGLU, TP_BF16, &plan));
    /* one workspace serves the 65-token prompt, the 64-token prompt and the
     * decode step */
    TP_CHECK(tp_plan_sizes(plan, 1, CAP, &packed_bytes, &ws_bytes));
    TP_CHECK(tp_plan_sizes(plan, 1, 1, NULL, &ws1));
    if (ws1 > ws_bytes) ws_bytes = ws1;

    /* full [out, in] weights Wq, Wk, Wv, Wo, Wgate, Wup, Wdown, then packed */
    for (k = 0; k < 7; ++k) {
        w[k] = device_bf16(rows[k] * cols[k], 0.05f, &rng);
        if (!w[k]) {
            fprintf(stderr, "weight %d: host or device allocation or copy failed\n", k);
            return 1;
        }
    }
    CU_CHECK(cudaMalloc(&packed, packed_bytes));
    TP_CHECK(tp_shard_weights(plan, w[0], w[1], w[2], w[3], w[4], w[5], w[6], packed, NULL));
    CU_CHECK(cudaDeviceSynchronize());
    for (k = 0; k < 7; ++k) CU_CHECK(cudaFree(w[k]));

    x = device_bf16((size_t)CAP * D, 1.0f, &rng);  /* 65 token rows */
    if (!x) {
        fprintf(stderr, "x: host or device allocation or copy failed\n");
        return 1;
    }
    CU_CHECK(cudaMalloc(&ws, ws_bytes));
    CU_CHECK(cudaMalloc(&kc, cache_bytes));
    CU_CHECK(cudaMalloc(&vc, cache_bytes));
    CU_CHECK(cudaMalloc((void**)&y_all, (size_t)CAP * D * sizeof(float)));
    CU_CHECK(cudaMalloc((void**)&y_prompt, (size_t)T * D * sizeof(float)));
    CU_CHECK(cudaMalloc((void**)&y_tok, (size_t)D * sizeof(float)));

    /* all 65 tokens as one causal prompt, no cache */
    TP_CHECK(tp_block_forward(plan, x, 1, CAP, 1, NULL, NULL, 0, 0, packed, ws, ws_bytes, y_all, NULL));
    /* the first 64 as a prompt that fills the cache, then token 64 decoded */
    TP_CHECK(tp_block_forward(plan, x, 1, T, 1, kc, vc, CAP, 0, packed, ws, ws_bytes, y_prompt, NULL));
    TP_CHECK(tp_block_forward(plan, (const char*)x + (size_t)T * D * sizeof(uint16_t), 1, 1, 1, kc, vc, CAP, T,
                              packed, ws, ws_bytes, y_tok, NULL));
    TP_CHECK(tp_sync_status(NULL));

    CU_CHECK(cudaMemcpy(h_all, y_all, sizeof h_all, cudaMemcpyDeviceToHost));
    CU_CHECK(cudaMemcpy(h_prompt, y_prompt, sizeof h_prompt, cudaMemcpyDeviceToHost));
    CU_CHECK(cudaMemcpy(h_tok, y_tok, sizeof h_tok, cudaMemcpyDeviceToHost));
    /* rows 0..63 of the cached prompt, then the decoded row 64, against the
     * 65-token prompt */
    for (i = 0; i < (size_t)CAP * D; ++i) {
        const double g = i < (size_t)T * D ? h_prompt[i] : h_tok[i - (size_t)T * D];
        const double r = h_all[i], e = fabs(g - r);
        if (!isfinite(g) || !isfinite(r)) {
            fprintf(stderr, "non-finite output at %zu\n", i);
            return 1;
        }
        if (e > num) num = e;
        if (fabs(r) > den) den = fabs(r);
    }
    if (!(den > 0.0) || num / den > 2e-2) {
        fprintf(stderr, "cached prompt + decode vs one prompt: normwise error %.3e\n",
                den > 0.0 ? num / den : -1.0);
        return 1;
    }

    CU_CHECK(cudaFree(x));
    CU_CHECK(cudaFree(ws));
    CU_CHECK(cudaFree(kc));
    CU_CHECK(cudaFree(vc));
    CU_CHECK(cudaFree(y_all));
    CU_CHECK(cudaFree(y_prompt));
    CU_CHECK(cudaFree(y_tok));
    CU_CHECK(cudaFree(packed));
    tp_plan_destroy(plan);
    printf("ok\n");
    return 0;
}
