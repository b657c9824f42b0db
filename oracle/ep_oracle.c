/*
 * ep_oracle.c -- plain CPU oracle for routed MoE expert-parallel dispatch and
 * combine, with all W expert-parallel ranks held in host memory.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library. It shares no
 * code, header, table or helper with the CUDA library; the two meet only in
 * the seeded inputs they are both given.
 *
 * What it follows: vLLM "AllToAllBatchedPrepareAndFinalize" (page
 * fused_moe/prepare_finalize/alltoall_batched), methods `capacities`,
 * `prepare` and `finalize`. Every function below names the part of those
 * methods it restates. It is written as slow, obvious loops: no blocking, no
 * reordering beyond what the method states. The all_to_all_single exchange of
 * the page is a plain block transpose here, because all ranks share one
 * address space: recv[d][s] = send[s][d]. `oracle_scale_input` restates the
 * same method's apply_router_weight_on_input branch. `oracle_agrs` follows
 * vLLM's AgRsAll2AllManager (page device_communicators/all2all, `dispatch`
 * and `combine`: all_gatherv, then reduce_scatterv) with identity experts.
 *
 * Readings of points the page leaves open (each also listed in the design
 * notes of the repository):
 *   - every negative expert id is dropped (the code keeps ids >= 0; its
 *     comment speaks of -1 only);
 *   - an id >= E is an error: flagged, and the pair is dropped;
 *   - a repeated id inside one token row is an error: flagged, and the later
 *     occurrence is dropped (the page would overflow its pick column);
 *   - the columns of a token's experts on one destination follow top-k order
 *     (the page sorts with an unstable argsort; its comment asks for the
 *     k-th expert in column k);
 *   - combine folds a token's experts in top-k order in fp32, one product and
 *     one sum per step, each rounded on its own (the page's finalize forms the
 *     weighted rows as an fp32 tensor before it accumulates them, so a product
 *     is rounded before it is added: no fused multiply-add), rounded once to
 *     the output type. A hand-derived golden case pins both the separate
 *     roundings and the top-k order of the fold. The page sums
 *     per-destination partials in fp32, rounds them to the activation type
 *     and sums those in the output type; `oracle_combine_pagemode` restates
 *     that two-stage form so tests can show both agree within tolerance;
 *   - in the AgRs route each rank applies only its own experts (the expert
 *     map of the fused-MoE layer), rounds its output to bf16, and the
 *     reduce-scatter sums the ranks' outputs in ascending rank order (each
 *     sum rounded for bf16 output, fp32 sums for fp32 output).
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (no FMA contraction, so each
 * product and each sum rounds on its own, as the fold above states). A second
 * build with -fopenmp serves only to time the oracle on all host cores: its
 * pragmas split the row copies and the combine over independent (rank, rank),
 * expert or token blocks. Every output element is still computed by one thread
 * in the order written here, so both builds give identical results; without
 * -fopenmp the pragmas are ignored.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Error kinds, OR-ed into *err. */
#define OR_ERR_EXPERT_ID 1u  /* an id >= E */
#define OR_ERR_DUPLICATE 2u  /* an id repeated within one token row */
#define OR_ERR_CAPACITY 4u   /* num_tokens[r] outside [0, Tm], or an expert over expert_cap */

static int imin(int a, int b) { return a < b ? a : b; }

/* capacities(topk) of the page: token slots per rank, expert slots per token,
 * rows per expert. */
void oracle_capacities(int W, int E, int K, int Tm, int *tok_cap, int *slots, int *expert_cap) {
    int e_local = E / W;
    *tok_cap = Tm;
    *slots = imin(K, e_local);
    *expert_cap = Tm * W;
}

/*
 * Step 1 and 2 of `prepare`, send side, one rank at a time: flatten the
 * (token, expert) pairs, drop the padding ones, find each pair's destination
 * rank d = expert / e_local, give each (d, token) group one slot on d in token
 * order, and fill that slot's local expert ids and router weights, column c
 * holding the c-th of the token's experts that live on d.
 *
 * Outputs (all written in full):
 *   send_cnt  [W(s)][W(d)]          tokens of s that go to d
 *   send_tok  [W(s)][W(d)][Tm]      token held by each slot, -1 past the count
 *   send_eloc [W(s)][W(d)][Tm][S]   local expert id per column, -1 unused
 *   send_w    [W(s)][W(d)][Tm][S]   router weight per column, 0 unused
 *   send_k    [W(s)][W(d)][Tm][S]   top-k index of the pair in that column, -1 unused
 */
void oracle_route(int W, int E, int K, int Tm, const int32_t *num_tokens, const int32_t *ids,
                  const float *weights, int32_t *send_cnt, int32_t *send_tok, int32_t *send_eloc,
                  float *send_w, int32_t *send_k, uint32_t *err) {
    int e_local = E / W;
    int S = imin(K, e_local);
    size_t nslot = (size_t)W * W * Tm;
    for (size_t i = 0; i < (size_t)W * W; ++i) send_cnt[i] = 0;
    for (size_t i = 0; i < nslot; ++i) send_tok[i] = -1;
    for (size_t i = 0; i < nslot * S; ++i) {
        send_eloc[i] = -1;
        send_w[i] = 0.0f;
        send_k[i] = -1;
    }
    int32_t *kept = (int32_t *)malloc(sizeof(int32_t) * (size_t)(K > 0 ? K : 1));
    int32_t *slot_on = (int32_t *)malloc(sizeof(int32_t) * (size_t)W);
    int32_t *used_cols = (int32_t *)malloc(sizeof(int32_t) * (size_t)W);
    for (int s = 0; s < W; ++s) {
        int T = num_tokens ? num_tokens[s] : Tm;
        if (T < 0 || T > Tm) {
            *err |= OR_ERR_CAPACITY;
            T = T < 0 ? 0 : Tm;
        }
        for (int t = 0; t < T; ++t) {
            const int32_t *row = ids + ((size_t)s * Tm + t) * K;
            /* the pairs that take part, in top-k order */
            for (int k = 0; k < K; ++k) {
                int e = row[k];
                kept[k] = 0;
                if (e < 0) continue;
                if (e >= E) { *err |= OR_ERR_EXPERT_ID; continue; }
                int dup = 0;
                for (int k2 = 0; k2 < k; ++k2)
                    if (kept[k2] && row[k2] == e) dup = 1;
                if (dup) { *err |= OR_ERR_DUPLICATE; continue; }
                kept[k] = 1;
            }
            /* one slot per destination the token reaches */
            for (int d = 0; d < W; ++d) { slot_on[d] = -1; used_cols[d] = 0; }
            for (int k = 0; k < K; ++k) {
                if (!kept[k]) continue;
                int d = row[k] / e_local;
                if (slot_on[d] < 0) {
                    slot_on[d] = send_cnt[s * W + d]++;
                    send_tok[((size_t)s * W + d) * Tm + slot_on[d]] = t;
                }
            }
            /* the token's experts on each destination, column by column */
            for (int k = 0; k < K; ++k) {
                if (!kept[k]) continue;
                int d = row[k] / e_local;
                int col = used_cols[d]++;
                size_t at = (((size_t)s * W + d) * Tm + slot_on[d]) * S + col;
                send_eloc[at] = row[k] - d * e_local;
                send_w[at] = weights[((size_t)s * Tm + t) * K + k];
                send_k[at] = k;
            }
        }
    }
    free(kept);
    free(slot_on);
    free(used_cols);
}

/* The metadata all_to_all_single of `prepare`: rank d receives, from each s,
 * the count and the columns s built for d. */
void oracle_exchange_meta(int W, int E, int K, int Tm, const int32_t *send_cnt,
                          const int32_t *send_eloc, const float *send_w, int32_t *recv_cnt,
                          int32_t *recv_eloc, float *recv_w) {
    int S = imin(K, E / W);
    size_t blk = (size_t)Tm * S;
    for (int s = 0; s < W; ++s)
        for (int d = 0; d < W; ++d) {
            recv_cnt[d * W + s] = send_cnt[s * W + d];
            memcpy(recv_eloc + ((size_t)d * W + s) * blk, send_eloc + ((size_t)s * W + d) * blk,
                   blk * sizeof(int32_t));
            memcpy(recv_w + ((size_t)d * W + s) * blk, send_w + ((size_t)s * W + d) * blk,
                   blk * sizeof(float));
        }
}

/*
 * The delivery of `prepare` into the batched-experts layout, on each rank d:
 * walk the received slots in (source rank, slot) order and, inside a slot, its
 * columns in order; each column naming local expert j takes the next free row
 * of expert j. expert_num_tokens[d][j] is the row count.
 *
 * Outputs:
 *   expert_num_tokens [W(d)][e_local]
 *   row_src  [W(d)][e_local][Ecap]  packed (s * Tm + slot) of the received
 *                                   slot in each row, -1 past the count
 *   row_col  [W(d)][e_local][Ecap]  column of that slot, -1 past the count
 */
void oracle_deliver_meta(int W, int E, int K, int Tm, const int32_t *recv_cnt,
                         const int32_t *recv_eloc, int32_t *expert_num_tokens, int32_t *row_src,
                         int32_t *row_col, uint32_t *err) {
    int e_local = E / W;
    int S = imin(K, e_local);
    int Ecap = Tm * W;
    for (size_t i = 0; i < (size_t)E * Ecap; ++i) { row_src[i] = -1; row_col[i] = -1; }
    for (int d = 0; d < W; ++d) {
        int32_t *n = expert_num_tokens + (size_t)d * e_local;
        for (int j = 0; j < e_local; ++j) n[j] = 0;
        for (int s = 0; s < W; ++s) {
            for (int slot = 0; slot < recv_cnt[d * W + s]; ++slot) {
                for (int c = 0; c < S; ++c) {
                    int j = recv_eloc[(((size_t)d * W + s) * Tm + slot) * S + c];
                    if (j < 0) continue;
                    int row = n[j]++;
                    if (row >= Ecap) { *err |= OR_ERR_CAPACITY; continue; }
                    size_t at = ((size_t)d * e_local + j) * Ecap + row;
                    row_src[at] = s * Tm + slot;
                    row_col[at] = c;
                }
            }
        }
    }
}

/*
 * The combine context of `prepare`, token side: for each (rank s, token t,
 * top-k index k) the row of the batched layout that holds the pair, as the flat
 * index (d * e_local + j) * Ecap + row, or -1 for a pair that takes no part.
 * Built by joining the delivered rows with the send-side slot tables.
 */
void oracle_pair_rows(int W, int E, int K, int Tm, const int32_t *expert_num_tokens,
                      const int32_t *row_src, const int32_t *row_col, const int32_t *send_tok,
                      const int32_t *send_k, int32_t *pair_row) {
    int e_local = E / W;
    int S = imin(K, e_local);
    int Ecap = Tm * W;
    for (size_t i = 0; i < (size_t)W * Tm * K; ++i) pair_row[i] = -1;
    for (int d = 0; d < W; ++d)
        for (int j = 0; j < e_local; ++j)
            for (int row = 0; row < expert_num_tokens[d * e_local + j] && row < Ecap; ++row) {
                size_t at = ((size_t)d * e_local + j) * Ecap + row;
                int s = row_src[at] / Tm, slot = row_src[at] % Tm, c = row_col[at];
                int t = send_tok[((size_t)s * W + d) * Tm + slot];
                int k = send_k[(((size_t)s * W + d) * Tm + slot) * S + c];
                pair_row[((size_t)s * Tm + t) * K + k] = (int32_t)at;
            }
}

/* send_x[s][d][slot] = a1[s][token of the slot]: the pack of `prepare`. Rows
 * past the count are zero, as the page's zero-filled send buffer. `rb` is the
 * row size in bytes; a row may be the activation followed by extra payloads. */
void oracle_pack(int W, int Tm, size_t rb, const int32_t *send_cnt, const int32_t *send_tok,
                 const uint8_t *src_rows, uint8_t *send_x) {
    memset(send_x, 0, (size_t)W * W * Tm * rb);
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int s = 0; s < W; ++s)
        for (int d = 0; d < W; ++d)
            for (int slot = 0; slot < send_cnt[s * W + d]; ++slot) {
                int t = send_tok[((size_t)s * W + d) * Tm + slot];
                memcpy(send_x + (((size_t)s * W + d) * Tm + slot) * rb,
                       src_rows + ((size_t)s * Tm + t) * rb, rb);
            }
}

/* The payload all_to_all_single: recv_x[d][s] = send_x[s][d]. */
void oracle_exchange(int W, int Tm, size_t rb, const uint8_t *send_x, uint8_t *recv_x) {
    size_t blk = (size_t)Tm * rb;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int s = 0; s < W; ++s)
        for (int d = 0; d < W; ++d)
            memcpy(recv_x + ((size_t)d * W + s) * blk, send_x + ((size_t)s * W + d) * blk, blk);
}

/* Delivered rows, packed: out_rows holds the rows of every (d, j) in (d, j,
 * row) order, expert (d, j) starting at row_off[d * e_local + j]. Row (d, j,
 * row) is a copy of recv_x[d][s][slot] for the slot recorded in row_src. */
void oracle_deliver(int W, int E, int Tm, size_t rb, const int32_t *expert_num_tokens,
                    const int32_t *row_src, const uint8_t *recv_x, const int64_t *row_off,
                    uint8_t *out_rows) {
    int e_local = E / W;
    int Ecap = Tm * W;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int d = 0; d < W; ++d)
        for (int j = 0; j < e_local; ++j) {
            int n = expert_num_tokens[d * e_local + j];
            for (int row = 0; row < n && row < Ecap; ++row) {
                int32_t src = row_src[((size_t)d * e_local + j) * Ecap + row];
                int s = src / Tm, slot = src % Tm;
                memcpy(out_rows + (size_t)(row_off[d * e_local + j] + row) * rb,
                       recv_x + (((size_t)d * W + s) * Tm + slot) * rb, rb);
            }
        }
}

static float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round to bfloat16, nearest with ties to even (the IEEE default mode). */
static uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/*
 * `finalize`: out[s][t] = sum over the token's pairs k of w[s][t][k] times
 * the expert row that holds the pair, in fp32, rounded once to the output
 * type. The fold runs k = 0..K-1 in order, skipping pairs that take no part:
 * p = w * x (rounded), acc = acc + p (rounded). Tokens with no pair, and rows
 * at or past num_tokens, give zeros.
 *
 * Expert rows are read from a packed table: the row of flat index f = (d *
 * e_local + j) * Ecap + row sits at rows[(row_off[d * e_local + j] + row) *
 * h]. out_f32 selects a float32 output; else the output is bf16 bits.
 * tokens / n_tokens select a subset of flat token indices (s * Tm + t) to
 * compute; NULL computes every token. out is indexed by flat token index.
 */
void oracle_combine(int W, int E, int K, int Tm, int h, const int32_t *num_tokens,
                    const int32_t *pair_row, const float *weights, const uint16_t *rows,
                    const int64_t *row_off, int out_f32, void *out, const int64_t *tokens,
                    int64_t n_tokens) {
    int Ecap = Tm * W;
    (void)E;   /* a flat row index needs only Ecap to split */
    int64_t n = tokens ? n_tokens : (int64_t)W * Tm;
#pragma omp parallel
    {
    float *acc = (float *)malloc(sizeof(float) * (size_t)h);
#pragma omp for schedule(static)
    for (int64_t q = 0; q < n; ++q) {
        int64_t g = tokens ? tokens[q] : q;
        int s = (int)(g / Tm), t = (int)(g % Tm);
        int T = num_tokens ? num_tokens[s] : Tm;
        for (int i = 0; i < h; ++i) acc[i] = 0.0f;
        if (t < T) {
            for (int k = 0; k < K; ++k) {
                int32_t f = pair_row[g * K + k];
                if (f < 0) continue;
                float w = weights[g * K + k];
                const uint16_t *x = rows + (size_t)(row_off[f / Ecap] + f % Ecap) * h;
                for (int i = 0; i < h; ++i) {
                    float p = w * bf16_to_f32(x[i]);
                    acc[i] = acc[i] + p;
                }
            }
        }
        if (out_f32) {
            memcpy((float *)out + (size_t)g * h, acc, sizeof(float) * (size_t)h);
        } else {
            uint16_t *o = (uint16_t *)out + (size_t)g * h;
            for (int i = 0; i < h; ++i) o[i] = f32_to_bf16(acc[i]);
        }
    }
    free(acc);
    }
}

/*
 * The all-gather / reduce-scatter route of vLLM's AgRsAll2AllManager (page
 * device_communicators/all2all: `dispatch` gathers hidden states, top-k weights
 * and ids of all ranks with all_gatherv; `combine` reduce-scatters), with the
 * experts in between being the identity and each rank applying only its own
 * experts, as the fused-MoE layer does with an expert map:
 *   on rank d, for every gathered token g: y_d[g] = bf16( fp32 fold over the
 *   token's kept pairs k whose expert lives on d, in top-k order, of w_k * x_g )
 *   (zero if none);
 *   reduce-scatter: out[g] = sum over d = 0..W-1 of y_d[g], in the output type
 *   (bf16: every sum rounded; f32: fp32 sums).
 * Pairs are kept by the same rule as oracle_route (negative ids dropped, ids
 * >= E and repeats flagged and dropped). Tokens at or past num_tokens give 0.
 */
void oracle_agrs(int W, int E, int K, int Tm, int h, const int32_t *num_tokens,
                 const int32_t *ids, const float *weights, const uint16_t *a1, int out_f32,
                 void *out, uint32_t *err) {
    int e_local = E / W;
    float *yd = (float *)malloc(sizeof(float) * (size_t)h);
    float *acc = (float *)malloc(sizeof(float) * (size_t)h);
    int32_t *kept = (int32_t *)malloc(sizeof(int32_t) * (size_t)(K > 0 ? K : 1));
    for (int s = 0; s < W; ++s) {
        int T = num_tokens ? num_tokens[s] : Tm;
        if (T < 0 || T > Tm) {
            *err |= OR_ERR_CAPACITY;
            T = T < 0 ? 0 : Tm;
        }
        for (int t = 0; t < Tm; ++t) {
            size_t g = (size_t)s * Tm + t;
            for (int i = 0; i < h; ++i) acc[i] = 0.0f;
            if (t < T) {
                const int32_t *row = ids + g * K;
                for (int k = 0; k < K; ++k) {
                    int e = row[k];
                    kept[k] = 0;
                    if (e < 0) continue;
                    if (e >= E) { *err |= OR_ERR_EXPERT_ID; continue; }
                    int dup = 0;
                    for (int k2 = 0; k2 < k; ++k2)
                        if (kept[k2] && row[k2] == e) dup = 1;
                    if (dup) { *err |= OR_ERR_DUPLICATE; continue; }
                    kept[k] = 1;
                }
                for (int d = 0; d < W; ++d) {      /* every rank's expert output */
                    for (int i = 0; i < h; ++i) yd[i] = 0.0f;
                    for (int k = 0; k < K; ++k) {
                        if (!kept[k] || row[k] / e_local != d) continue;
                        float w = weights[g * K + k];
                        for (int i = 0; i < h; ++i) {
                            float p = w * bf16_to_f32(a1[g * h + i]);
                            yd[i] = yd[i] + p;
                        }
                    }
                    for (int i = 0; i < h; ++i) {    /* the reduce-scatter sum */
                        float y = bf16_to_f32(f32_to_bf16(yd[i]));
                        if (out_f32) acc[i] = acc[i] + y;
                        else acc[i] = bf16_to_f32(f32_to_bf16(acc[i] + y));
                    }
                }
            }
            if (out_f32) {
                memcpy((float *)out + g * h, acc, sizeof(float) * (size_t)h);
            } else {
                uint16_t *o = (uint16_t *)out + g * h;
                for (int i = 0; i < h; ++i) o[i] = f32_to_bf16(acc[i]);
            }
        }
    }
    free(yd);
    free(acc);
    free(kept);
}

/*
 * `prepare` with apply_router_weight_on_input (the page allows it for top_k == 1
 * only): a1 is multiplied by the router weight converted to the activation
 * type, a1 = a1 * topk_weights.to(a1.dtype), so each element becomes
 * bf16(x * bf16(w)); the weights carried on are then all one. rows are [n][h]
 * bf16 bits, weights [n].
 */
void oracle_scale_input(int64_t n, int h, const uint16_t *rows, const float *weights,
                        uint16_t *out) {
    for (int64_t g = 0; g < n; ++g) {
        float w = bf16_to_f32(f32_to_bf16(weights[g]));
        for (int i = 0; i < h; ++i) {
            float x = bf16_to_f32(rows[g * h + i]);
            out[g * h + i] = f32_to_bf16(x * w);
        }
    }
}

/*
 * `finalize` in the page's own two-stage form, kept for comparison: on each
 * rank d the pairs of each received slot are weighted and summed in fp32
 * (columns in order), the partial is rounded to bf16 (the activation type) for
 * the return all_to_all_single, and each token then sums its partials over
 * destinations in ascending order in the output type (bf16 sums rounded after
 * every add; f32 sums in fp32).
 */
void oracle_combine_pagemode(int W, int E, int K, int Tm, int h, const int32_t *send_cnt,
                             const int32_t *send_tok, const int32_t *send_eloc,
                             const float *send_w, const int32_t *recv_rows_of_slot,
                             const uint16_t *rows, const int64_t *row_off, int out_f32,
                             void *out) {
    /* recv_rows_of_slot[W(s)][W(d)][Tm][S]: the flat row (as in pair_row) of
     * each column of each send slot, -1 unused. */
    int e_local = E / W;
    int S = imin(K, e_local);
    int Ecap = Tm * W;
    float *part = (float *)malloc(sizeof(float) * (size_t)h);
    float *acc = (float *)malloc(sizeof(float) * (size_t)h);
    for (int s = 0; s < W; ++s)
        for (int t = 0; t < Tm; ++t) {
            for (int i = 0; i < h; ++i) acc[i] = 0.0f;
            for (int d = 0; d < W; ++d) {
                int slot = -1;
                for (int q = 0; q < send_cnt[s * W + d]; ++q)
                    if (send_tok[((size_t)s * W + d) * Tm + q] == t) slot = q;
                if (slot < 0) continue;
                for (int i = 0; i < h; ++i) part[i] = 0.0f;
                for (int c = 0; c < S; ++c) {
                    size_t at = (((size_t)s * W + d) * Tm + slot) * S + c;
                    if (send_eloc[at] < 0) continue;
                    int32_t f = recv_rows_of_slot[at];
                    const uint16_t *x = rows + (size_t)(row_off[f / Ecap] + f % Ecap) * h;
                    for (int i = 0; i < h; ++i) {
                        float p = bf16_to_f32(x[i]) * send_w[at];
                        part[i] = part[i] + p;
                    }
                }
                for (int i = 0; i < h; ++i) {
                    float pr = bf16_to_f32(f32_to_bf16(part[i]));
                    if (out_f32) acc[i] = acc[i] + pr;
                    else acc[i] = bf16_to_f32(f32_to_bf16(acc[i] + pr));
                }
            }
            if (out_f32) {
                memcpy((float *)out + ((size_t)s * Tm + t) * h, acc, sizeof(float) * (size_t)h);
            } else {
                uint16_t *o = (uint16_t *)out + ((size_t)s * Tm + t) * h;
                for (int i = 0; i < h; ++i) o[i] = f32_to_bf16(acc[i]);
            }
        }
    free(part);
    free(acc);
}
