/*
 * c_abi_client.c -- the EP library driven from plain C, through include/ep.h and
 * the CUDA runtime API only (no Python, no PyTorch): size and create a context
 * over a workspace this program allocates, dispatch W ranks' tokens, run the
 * combine on the dispatched rows (identity experts) and check the results on
 * the host.
 *
 * Router weights are powers of two that sum to one (1/2, 1/4, ..., 2^-(K-1),
 * 2^-(K-1)), so every product and sum of the combine's fp32 fold is exact and
 * each routed token must come back bit for bit; a token whose ids are all -1
 * must come back as zeros. Each expert's row count must equal the number of
 * (token, expert) pairs that chose it.
 *
 * Exit status 0 and "c client ok" on success; anything else names the failure.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "ep.h"

#define CHECK_CUDA(x)                                                              \
    do {                                                                           \
        cudaError_t e_ = (x);                                                      \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));               \
            return 2;                                                              \
        }                                                                          \
    } while (0)

#define CHECK_EP(x)                                                                \
    do {                                                                           \
        int r_ = (x);                                                              \
        if (r_ != EP_OK) {                                                         \
            fprintf(stderr, "%s: %s (%d)\n", #x, ep_error_string(r_), r_);         \
            return 3;                                                              \
        }                                                                          \
    } while (0)

static uint64_t lcg_state = 88172645463325252ull;
static uint32_t lcg(void) {
    lcg_state = lcg_state * 6364136223846793005ull + 1442695040888963407ull;
    return (uint32_t)(lcg_state >> 33);
}

/* a bf16 bit pattern of a finite value in about [-2, 2): sign, exponent 126 or 127, random mantissa */
static uint16_t random_bf16(void) {
    const uint32_t r = lcg();
    return (uint16_t)(((r & 1u) << 15) | ((126u + ((r >> 1) & 1u)) << 7) | ((r >> 2) & 0x7Fu));
}

int main(void) {
    ep_config_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.W = 4;
    cfg.E = 32;
    cfg.top_k = 4;
    cfg.max_tokens = 96;
    cfg.hidden = 256;
    cfg.x_dtype = EP_BF16;
    const int W = cfg.W, E = cfg.E, K = cfg.top_k, Tm = cfg.max_tokens, h = cfg.hidden;

    int32_t tok_cap = 0, slots = 0, ecap = 0;
    size_t ws_bytes = 0;
    CHECK_EP(ep_capacities(&cfg, &tok_cap, &slots, &ecap));
    CHECK_EP(ep_workspace_bytes(&cfg, &ws_bytes));
    const int e_local = E / W;
    const size_t n_tok = (size_t)W * Tm;

    /* host inputs */
    uint16_t *a1 = (uint16_t *)malloc(n_tok * h * sizeof(uint16_t));
    int32_t *ids = (int32_t *)malloc(n_tok * K * sizeof(int32_t));
    float *w = (float *)malloc(n_tok * K * sizeof(float));
    uint16_t *out = (uint16_t *)malloc(n_tok * h * sizeof(uint16_t));
    int32_t *ent = (int32_t *)malloc((size_t)E * sizeof(int32_t));
    int32_t *want_ent = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    if (!a1 || !ids || !w || !out || !ent || !want_ent) return 4;
    for (size_t i = 0; i < n_tok * h; ++i) a1[i] = random_bf16();
    for (size_t g = 0; g < n_tok; ++g) {
        const int padding = (g % 17) == 5;   /* some tokens choose no expert */
        for (int k = 0; k < K; ++k) {
            int e = -1;
            if (!padding) {
                int fresh = 0;
                while (!fresh) {   /* distinct experts per token */
                    e = (int)(lcg() % (uint32_t)E);
                    fresh = 1;
                    for (int k2 = 0; k2 < k; ++k2) fresh &= ids[g * K + k2] != e;
                }
                want_ent[e] += 1;
            }
            ids[g * K + k] = e;
            w[g * K + k] = k + 1 < K ? 1.0f / (float)(1 << (k + 1)) : 1.0f / (float)(1 << (K - 1));
        }
    }

    /* device buffers: the library allocates nothing, the caller owns them all */
    void *d_ws = NULL, *d_a1 = NULL, *d_b = NULL, *d_out = NULL;
    int32_t *d_ids = NULL, *d_ent = NULL;
    float *d_w = NULL;
    CHECK_CUDA(cudaMalloc(&d_ws, ws_bytes));
    CHECK_CUDA(cudaMalloc(&d_a1, n_tok * h * 2));
    CHECK_CUDA(cudaMalloc((void **)&d_ids, n_tok * K * 4));
    CHECK_CUDA(cudaMalloc((void **)&d_w, n_tok * K * 4));
    CHECK_CUDA(cudaMalloc(&d_b, (size_t)W * e_local * ecap * h * 2));   /* [W][e_local][Ecap][h] */
    CHECK_CUDA(cudaMalloc((void **)&d_ent, (size_t)E * 4));
    CHECK_CUDA(cudaMalloc(&d_out, n_tok * h * 2));
    CHECK_CUDA(cudaMemcpy(d_a1, a1, n_tok * h * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_ids, ids, n_tok * K * 4, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_w, w, n_tok * K * 4, cudaMemcpyHostToDevice));

    ep_ctx_t *ctx = NULL;
    CHECK_EP(ep_ctx_create(&cfg, d_ws, ws_bytes, &ctx));
    /* combine before dispatch is refused by the state rule */
    if (ep_combine(ctx, d_b, EP_BF16, d_out, NULL) != EP_ERR_STATE) {
        fprintf(stderr, "combine before dispatch was not refused\n");
        return 5;
    }
    CHECK_EP(ep_dispatch(ctx, d_a1, NULL, d_ids, d_w, NULL, d_b, NULL, d_ent, EP_PATH_FUSED, NULL));
    CHECK_EP(ep_combine(ctx, d_b, EP_BF16, d_out, NULL));   /* identity experts: expert_out = b_a1 */
    CHECK_EP(ep_status(ctx, NULL));
    CHECK_CUDA(cudaMemcpy(out, d_out, n_tok * h * 2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(ent, d_ent, (size_t)E * 4, cudaMemcpyDeviceToHost));

    for (int e = 0; e < E; ++e)
        if (ent[e] != want_ent[e]) {
            fprintf(stderr, "expert %d: %d rows, want %d\n", e, ent[e], want_ent[e]);
            return 6;
        }
    for (size_t g = 0; g < n_tok; ++g) {
        const int padding = ids[g * K] < 0;
        for (int i = 0; i < h; ++i) {
            const uint16_t want = padding ? 0 : a1[g * h + i];
            if (out[g * h + i] != want) {
                fprintf(stderr, "token %zu element %d: 0x%04x, want 0x%04x\n", g, i, out[g * h + i], want);
                return 7;
            }
        }
    }

    CHECK_EP(ep_ctx_destroy(ctx));
    cudaFree(d_ws);
    cudaFree(d_a1);
    cudaFree(d_ids);
    cudaFree(d_w);
    cudaFree(d_b);
    cudaFree(d_ent);
    cudaFree(d_out);
    free(a1);
    free(ids);
    free(w);
    free(out);
    free(ent);
    free(want_ent);
    printf("c client ok: %d ranks, %d experts, top_k %d, %d tokens per rank, %u workspace bytes\n", W, E, K,
           Tm, (unsigned)ws_bytes);
    return 0;
}
