/*
 * ep.h -- routed Mixture-of-Experts expert-parallel (EP) dispatch and combine
 * on one GB300 GPU, with all W expert-parallel ranks simulated as blocks of
 * that GPU's memory. The all-to-all exchange of a multi-GPU deployment becomes
 * a permutation between rank blocks in HBM.
 *
 * What is computed follows vLLM "AllToAllBatchedPrepareAndFinalize" (page
 * fused_moe/prepare_finalize/alltoall_batched): `capacities`, `prepare`
 * (dispatch) and `finalize` (combine). The sizing, state rules and
 * multi-payload dispatch follow FlashInfer "MoE All-to-All Operations
 * (Throughput Backend)" (page flashinfer/comm/trtllm_moe_alltoall.py:
 * `moe_a2a_get_workspace_size_per_rank`, `MoeAlltoAll.dispatch/combine`,
 * `_A2AState`). The all-gather / reduce-scatter route (ep_agrs) follows vLLM's
 * AgRsAll2AllManager (page device_communicators/all2all).
 *
 * Conventions for every entry point:
 *   - Return value: EP_OK (0) or a negative EP_ERR_* code; nothing else
 *     (ep_error_string, which returns a message, is the one exception).
 *   - "device" pointers are CUDA global-memory addresses of the current device;
 *     "host" pointers are ordinary process memory. The library never allocates
 *     device memory: the caller owns every buffer, including the workspace,
 *     and keeps it alive while the context uses it.
 *   - Work is enqueued on the caller's stream (a cudaStream_t passed as void*,
 *     NULL = the legacy default stream) with no host synchronisation, except in
 *     ep_status and ep_kernel_times, which synchronise.
 *   - Layouts are dense, row-major, with a leading rank dimension [W]:
 *       a1            [W][Tm][h]            x_dtype (bf16; or fp8 / packed fp4 bytes)
 *       topk_ids      [W][Tm][K]            int32, negative = no expert
 *       topk_weights  [W][Tm][K]            float32
 *       num_tokens    [W]                   int32 (rank r holds tokens 0..num_tokens[r]-1)
 *       b_a1          [W][e_local][Ecap][h] x_dtype, the batched-experts layout
 *       expert_num_tokens [W][e_local]      int32
 *       extra_in[i]   [W][Tm][extra_row_bytes[i]]        opaque bytes
 *       extra_out[i]  [W][e_local][Ecap][extra_row_bytes[i]]
 *       expert_out    like b_a1;  out  [W][Tm][h] bf16 or float32
 *     with Tm = max_tokens, e_local = E / W, Ecap = Tm * W (rows per expert).
 *   - Alignment: a1, b_a1, expert_out, out and every extra buffer 16 bytes;
 *     the workspace 256 bytes; the others 4 bytes.
 *   - A context is used by one host thread at a time. Its dispatch and combine
 *     are ordered by the stream they are given; running one context on two
 *     streams at once races on its workspace.
 *   - Several devices: work goes to the device current when a call is made,
 *     which must be the device of its buffers (a context's workspace binds it
 *     to one device). The kernels' raised shared-memory limits are kept per
 *     (kernel, device) under a lock, so one process may drive several GPUs
 *     from one or several host threads.
 */
#ifndef EP_H
#define EP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ limits */
#define EP_MAX_W 64       /* simulated ranks */
#define EP_MAX_E 1024     /* experts in total */
#define EP_MAX_TOPK 16    /* experts per token */
#define EP_MAX_EXTRA 4    /* extra payloads per dispatch */

/* ------------------------------------------------------------ status codes */
#define EP_OK 0
#define EP_ERR_INVALID_ARG -1 /* bad config, null or misaligned pointer, bad path or dtype */
#define EP_ERR_CAPACITY -2    /* a rank's num_tokens outside [0, max_tokens] (found on the device) */
#define EP_ERR_STATE -3       /* dispatch twice without combine, or combine before dispatch */
#define EP_ERR_EXPERT_ID -4   /* an expert id >= E (found on the device; the pair is dropped) */
#define EP_ERR_DUPLICATE -5   /* an expert id repeated in one token row (found on the device;
                                 the later occurrence is dropped) */
#define EP_ERR_TIMEOUT -6     /* a bounded device-side wait expired; outputs of that call are invalid */
#define EP_ERR_WORKSPACE -7   /* workspace too small or misaligned for the config or the path */
#define EP_ERR_CUDA -8        /* a CUDA runtime call or kernel launch failed */

/* ------------------------------------------------------------------- dtypes */
#define EP_BF16 1  /* activation rows / outputs: 2 bytes per element */
#define EP_F32 2   /* combine output: 4 bytes per element */
#define EP_FP8 3   /* dispatched activation rows as 1-byte elements (e.g. fp8 e4m3); opaque here */
#define EP_FP4X2 4 /* dispatched activation rows as packed 4-bit pairs (h/2 bytes); opaque here */

/* ----------------------------------------------------------- dispatch paths */
#define EP_PATH_FUSED 0   /* a1 -> b_a1 directly, each token row read once */
#define EP_PATH_SENDBUF 1 /* pack into send buffers, exchange rank blocks, deliver */

/* ---------------------------------------------------------------- flags */
#define EP_FLAG_ZERO_PAD 1u /* dispatch also zeroes b_a1 / extra_out rows at or past
                               expert_num_tokens (the page zero-fills them) and resets the
                               received-slot metadata of slots past the counts to the page's
                               fill (local id -1, weight 0, row -1); otherwise those rows and
                               slots are left as they were */
#define EP_FLAG_SENDBUF 2u  /* size the workspace for EP_PATH_SENDBUF as well */
#define EP_FLAG_WEIGHT_ON_INPUT 4u /* apply_router_weight_on_input of `prepare`: top_k must be
                                      1; dispatch delivers bf16(a1 * bf16(w)) and carries unit
                                      weights, so combine returns the expert row unweighted */

typedef struct ep_config {
    int32_t W;          /* simulated expert-parallel ranks, 1..EP_MAX_W */
    int32_t E;          /* experts in total, a multiple of W, <= EP_MAX_E */
    int32_t top_k;      /* experts per token, 1..min(E, EP_MAX_TOPK) */
    int32_t max_tokens; /* token slots per rank (Tm), >= 1 */
    int32_t hidden;     /* h, elements per row; 2*h and the dispatched row bytes must be
                           multiples of 16 */
    int32_t x_dtype;    /* dispatched a1 / b_a1 element type: EP_BF16, EP_FP8 or EP_FP4X2.
                           Quantised rows (the page's one-sided sizing: nvfp4 h/2 bytes plus
                           fp8 block scales) travel as opaque bytes; scales go as extra
                           payloads. expert_out and out of combine stay bf16 / f32. */
    int32_t n_extra;    /* extra payloads, 0..EP_MAX_EXTRA */
    int32_t extra_row_bytes[EP_MAX_EXTRA]; /* each a positive multiple of 16 */
    uint32_t flags;     /* EP_FLAG_* */
} ep_config_t;

typedef struct ep_ctx ep_ctx_t;

/*
 * ep_capacities -- `capacities(topk)` of AllToAllBatchedPrepareAndFinalize:
 * token slots per rank (*tok_cap = max_tokens), expert slots per token
 * (*slots_per_token = min(top_k, e_local)) and rows per expert (*expert_cap =
 * max_tokens * W). All pointers are host pointers. EP_ERR_INVALID_ARG for an
 * invalid config or a null pointer. Touches no GPU.
 */
int ep_capacities(const ep_config_t *cfg, int32_t *tok_cap, int32_t *slots_per_token,
                  int32_t *expert_cap);

/*
 * ep_workspace_bytes -- device workspace a context needs for cfg (host
 * pointers in and out). Sub-buffers are padded to 256 bytes, as
 * `moe_a2a_get_workspace_size_per_rank` pads its regions. It holds the
 * routing metadata (`prepare`'s combine context) and, with EP_FLAG_SENDBUF, the
 * send and receive rank blocks. Touches no GPU.
 */
int ep_workspace_bytes(const ep_config_t *cfg, size_t *bytes);

/*
 * ep_ctx_create -- bind a context to cfg and to a caller-owned device
 * workspace of at least ep_workspace_bytes(cfg) bytes (256-byte aligned).
 * Counterpart of FlashInfer `MoeAlltoAll.__init__` (page
 * flashinfer/comm/trtllm_moe_alltoall.py), which sizes a workspace per rank,
 * takes it from `MoeAlltoAll.get_workspace` (a per-process cache,
 * `_WORKSPACE_CACHE`, keyed by size, rank, EP size and max tokens) and starts
 * in the idle phase of `_A2AState`. Here the caller allocates and owns the
 * workspace (the library allocates no device memory) and may keep one per
 * configuration as that cache does. The context (host memory, freed by
 * ep_ctx_destroy) keeps pointers only and starts idle. The workspace is
 * initialised on first use, on the first dispatch's stream. Touches no GPU.
 * EP_ERR_INVALID_ARG for a bad config or null pointer, EP_ERR_WORKSPACE for a
 * small or misaligned workspace.
 */
int ep_ctx_create(const ep_config_t *cfg, void *d_workspace, size_t workspace_bytes,
                  ep_ctx_t **out);

/*
 * ep_ctx_destroy -- free the host context (not the workspace, which the
 * caller owns). NULL is a no-op. The FlashInfer page keeps its workspaces in
 * `MoeAlltoAll._WORKSPACE_CACHE` for the life of the process and drops one only
 * in `_reset_workspace`; here the caller frees the workspace once every
 * context bound to it is destroyed and its last stream work has finished.
 * Touches no GPU.
 */
int ep_ctx_destroy(ep_ctx_t *ctx);

/*
 * ep_dispatch -- `prepare` of AllToAllBatchedPrepareAndFinalize for all W
 * ranks at once, plus FlashInfer `MoeAlltoAll.dispatch`'s extra payloads.
 *
 * For every rank s and token t < num_tokens[s]: pairs with a negative id take
 * no part; each other pair (t, k) goes to rank d = id / e_local, local expert
 * j = id % e_local. A token goes to each rank it reaches once, in a slot
 * numbered in token order; the slot carries the token's local ids and router
 * weights on that rank, the k-th expert there in column k. Each rank d then
 * writes, for sources s ascending and slots ascending, one row per column into
 * b_a1[d][j][next free row of j], and the matching extra_out rows;
 * expert_num_tokens[d][j] counts them. No expert can overflow Ecap.
 *
 *   a1, topk_ids, topk_weights : device, read-only; may be reused once the
 *                                dispatch has run on the stream (the router
 *                                weights are copied into the workspace).
 *   num_tokens : device [W] or NULL (= max_tokens for every rank).
 *   extra_in / extra_out : HOST arrays of n_extra DEVICE pointers (NULL when
 *                          n_extra is 0).
 *   b_a1, extra_out[i], expert_num_tokens : device, written.
 *   path : EP_PATH_FUSED or EP_PATH_SENDBUF (needs EP_FLAG_SENDBUF).
 *
 * Host-side errors (returned, nothing enqueued): EP_ERR_INVALID_ARG,
 * EP_ERR_STATE (a dispatch already awaits its combine), EP_ERR_WORKSPACE,
 * EP_ERR_CUDA. Device-side errors (EP_ERR_EXPERT_ID, EP_ERR_DUPLICATE,
 * EP_ERR_CAPACITY, EP_ERR_TIMEOUT) are recorded in the workspace and returned
 * by ep_status.
 */
int ep_dispatch(ep_ctx_t *ctx, const void *a1, const int32_t *num_tokens,
                const int32_t *topk_ids, const float *topk_weights,
                const void *const *extra_in, void *b_a1, void *const *extra_out,
                int32_t *expert_num_tokens, int32_t path, void *stream);

/*
 * ep_combine -- `finalize` of AllToAllBatchedPrepareAndFinalize for all ranks:
 * out[s][t] = sum over the token's pairs k of w[s][t][k] * expert_out[d][j][row]
 * of the row the pair was delivered to, folded in fp32 in top-k order (one
 * rounded product and one rounded sum per pair) and rounded once to out_dtype
 * (EP_BF16 nearest-even, or EP_F32). Tokens with no pair and rows at or past
 * num_tokens[s] are written as zeros.
 *
 *   expert_out : device, layout of b_a1 (it may be b_a1 itself).
 *   out        : device [W][Tm][h] of out_dtype, written.
 *
 * Needs a preceding ep_dispatch on this context (EP_ERR_STATE otherwise, as
 * `MoeAlltoAll.combine` asserts); the context returns to idle afterwards.
 */
int ep_combine(ep_ctx_t *ctx, const void *expert_out, int32_t out_dtype, void *out,
               void *stream);

/*
 * ep_combine_two_stage -- `finalize` of AllToAllBatchedPrepareAndFinalize in
 * the page's own two-stage rounding, for comparison with ep_combine. Stage 1,
 * on each receiving rank d: for every received slot, sum its columns' expert
 * rows weighted by the router weights in fp32 (columns in order) and round the
 * partial to bf16 -- the payload the page returns with all_to_all_single.
 * Stage 2, on each sending rank s: out[s][t] = the sum of the token's partials
 * over the ranks it went to, ranks ascending, in out_dtype (EP_BF16: each sum
 * rounded to bf16; EP_F32: fp32 sums). It moves about twice the bytes of
 * ep_combine and rounds more often; results stay within the page's bound of
 * the single fold (2^-6 * sum_k |w_k x_k| element-wise).
 *
 * Needs a workspace sized with EP_FLAG_SENDBUF (its receive blocks hold the
 * stage-1 partials; EP_ERR_WORKSPACE otherwise) and a preceding ep_dispatch
 * (EP_ERR_STATE otherwise); arguments and state rule as ep_combine.
 */
int ep_combine_two_stage(ep_ctx_t *ctx, const void *expert_out, int32_t out_dtype, void *out,
                         void *stream);

/*
 * ep_status -- synchronise the stream, then return and clear the first
 * device-side error recorded since the last call (EP_OK if none), or
 * EP_ERR_CUDA if the stream reports a CUDA error.
 *
 * The errors it reports are the checks FlashInfer's `MoeAlltoAll.dispatch` and
 * `MoeAlltoAll.combine` make as asserts (runtime token count at most
 * max_num_tokens; page flashinfer/comm/trtllm_moe_alltoall.py) plus the id
 * checks the vLLM `prepare` leaves undefined (ids >= E, repeated ids; page
 * fused_moe/prepare_finalize/alltoall_batched). Because those inputs live on
 * the device, the checks run there and land in a status word. Reading it
 * synchronises the host with the stream, which `prepare`'s rule of
 * fixed-size collectives with no host sync avoids on purpose: ep_status is
 * the one deliberate exception, for tests and debugging, and no other entry
 * point calls it.
 */
int ep_status(ep_ctx_t *ctx, void *stream);

/*
 * ep_ctx_reset -- return the context to idle, dropping a dispatch that will
 * not be combined. Counterpart of FlashInfer `MoeAlltoAll._reset_workspace`
 * (page flashinfer/comm/trtllm_moe_alltoall.py), which the page keeps for
 * testing: it synchronises, forgets the cached workspace and leaves the object
 * unusable. Here the context stays usable and the workspace stays the
 * caller's: only the `_A2AState` phase goes back to idle. Host only; touches
 * no GPU and enqueues nothing.
 */
int ep_ctx_reset(ep_ctx_t *ctx);

/*
 * Routing metadata kept in the workspace (device pointers; valid after a
 * dispatch has run). Filled by ep_get_metadata, which touches no GPU. It is
 * this library's counterpart of FlashInfer's metainfo accessors
 * (`MoeAlltoAll._init_constants`, `moe_a2a_get_metainfo_index_pairs`, page
 * flashinfer/comm/trtllm_moe_alltoall.py), which name offsets into the
 * workspace "for testing/debugging". The arrays are the combine context vLLM's
 * `prepare` builds and `finalize` consumes (page
 * fused_moe/prepare_finalize/alltoall_batched): per-destination counts, the
 * received slots' local expert ids and weights, and where each pair landed.
 *   send_cnt  [W(s)][W(d)]          tokens rank s sends to rank d
 *   pair_row  [W][Tm][K]            flat b_a1 row (d*e_local+j)*Ecap+row of each pair, -1
 *   pair_w    [W][Tm][K]            router weight of each kept pair, 0 otherwise
 *   pair_send [W][Tm][K]            send_x row (s*W+d)*Tm+slot for the first pair of a
 *                                   token on each rank, -1 otherwise
 *   recv_eloc [W(d)][W(s)][Tm][S]   local expert id per received slot and column, -1
 *   recv_w    [W(d)][W(s)][Tm][S]   router weight per received slot and column, 0
 *   recv_row  [W(d)][W(s)][Tm][S]   row of that column within its expert, -1
 *   send_x / recv_x [W][W][Tm][row_bytes]  rank blocks of the send-buffer path, or NULL
 * Entries of slots at or past send_cnt are unspecified.
 */
typedef struct ep_metadata {
    int32_t *send_cnt;
    int32_t *pair_row;
    float *pair_w;
    int32_t *pair_send;
    int32_t *recv_eloc;
    float *recv_w;
    int32_t *recv_row;
    void *send_x;
    void *recv_x;
    int32_t slots_per_token; /* S */
    int32_t expert_cap;      /* Ecap */
    int32_t row_bytes;       /* bytes of one send-buffer row: 2*h + sum of extra_row_bytes */
    int32_t reserved;
} ep_metadata_t;

/* ep_get_metadata -- fill *out (host) with the device addresses above. EP_ERR_INVALID_ARG
 * for a null pointer. Host only. */
int ep_get_metadata(const ep_ctx_t *ctx, ep_metadata_t *out);

/* ep_error_string -- static text for a status code. */
const char *ep_error_string(int code);

/* ------------------------------------------------------- tuning and checks */
#define EP_OPT_WAIT_LIMIT_NS 1   /* bound of every device-side wait, ns (default 2e9) */
#define EP_OPT_KERNEL_TIMING 2   /* 1: record CUDA events around every kernel */
#define EP_OPT_PDL 3             /* 1: programmatic dependent launch between kernels (default 0) */
#define EP_OPT_MOVE_CTAS_PER_SM 4 /* row-mover CTAs per SM (default 1) */
#define EP_OPT_MOVE_PIPES 5      /* row-mover pipelines (warps) per CTA, 1..8; in the
                                    one-launch fused dispatch, the warps of its 256 that move
                                    rows once routing is done. -1 (default) = chosen per
                                    problem (EP_OPT_MOVE_* together: by top_k and row size) */
#define EP_OPT_FAULT_SKIP_PUBLISH 6 /* test hook: the routing tile with this ticket never
                                       publishes, so its successors' waits run out and
                                       report EP_ERR_TIMEOUT; -1 (default) = off */
#define EP_OPT_COMBINE_CTAS_PER_SM 7 /* combine CTAs per SM (default 0: for top_k above 4 one wave
                                        of at most 3 per SM, or of all that fit when a wave covers
                                        the work in at most 4 rounds; for top_k up to 4 a grid of
                                        16 per SM) */
#define EP_OPT_MOVE_CHUNK_BYTES 8 /* row-mover unit: rows split into chunks of at least this
                                     many bytes (multiple of 16; 0 = whole rows; -1 = default,
                                     chosen per problem) */
#define EP_OPT_MOVE_MAX_STAGES 9  /* row-mover stages per pipeline, at most (2..32; -1 = default,
                                     chosen per problem) */
#define EP_OPT_FUSED_DISPATCH 10  /* 1 (default): the fused path routes and moves rows in one
                                     persistent launch, movement starting as tiles finish */
#define EP_OPT_ROUTE_CTAS 11      /* one-launch fused dispatch: how many CTAs route (the first
                                     to start; the others move rows from the outset);
                                     0 = every CTA routes first; -1 (default) = chosen per
                                     problem: 0 up to 32 routing tiles, else enough routers to
                                     stay ahead of the row movers, at least 32 (-1..4096) */
#define EP_OPT_SMALL_DISPATCH 12  /* fused path on a small batch (W * max_tokens * top_k at most
                                     16384, at most 32 token slots per SM): one launch in which
                                     every CTA counts its own tokens' prefix from the earlier
                                     tokens' ids, with no waiting between CTAs. -1 (default) =
                                     used whenever the batch qualifies, 0 = never, 1 = as -1 */

/* ep_set_option -- set one EP_OPT_* value (host only). EP_ERR_INVALID_ARG for an unknown option or value. */
int ep_set_option(ep_ctx_t *ctx, int32_t option, int64_t value);

/* Kernel kinds counted by ep_kernel_times. */
#define EP_K_ROUTE 0
#define EP_K_MOVE_FUSED 1
#define EP_K_PACK 2
#define EP_K_EXCHANGE 3
#define EP_K_DELIVER 4
#define EP_K_COMBINE 5
#define EP_K_ZERO_PAD 6
#define EP_K_COMBINE_TWO_STAGE 7
#define EP_K_DISPATCH_FUSED 8   /* routing + fused row movement in one launch */
#define EP_K_DISPATCH_SMALL 9   /* the same for a small batch, without waits between CTAs */
#define EP_K_COUNT 10

typedef struct ep_kernel_times {
    int64_t launches[EP_K_COUNT]; /* kernels launched, per kind, since the last read */
    double total_ms[EP_K_COUNT];  /* summed CUDA-event durations (EP_OPT_KERNEL_TIMING on) */
    int64_t timed[EP_K_COUNT];    /* launches those durations cover */
} ep_kernel_times_t;

/* ep_kernel_times -- read and reset the per-kernel launch counts and, with
 * EP_OPT_KERNEL_TIMING on, the event durations (waits for the events). */
int ep_kernel_times(ep_ctx_t *ctx, ep_kernel_times_t *out);

/* ------------------------------------------------- routing without allocation */
#define EP_ERR_SCRATCH_LIMIT -9 /* the problem needs more than EP_STATIC_SCRATCH_BYTES of scratch */
#define EP_STATIC_SCRATCH_BYTES (4u << 20)

/* Device output buffers of ep_route_static (layouts as in ep_metadata_t). */
typedef struct ep_route_outputs {
    int32_t *send_cnt;          /* [W(s)][W(d)] */
    int32_t *pair_row;          /* [W][Tm][K] */
    float *pair_w;              /* [W][Tm][K] */
    int32_t *pair_send;         /* [W][Tm][K] */
    int32_t *recv_eloc;         /* [W(d)][W(s)][Tm][S] */
    float *recv_w;              /* [W(d)][W(s)][Tm][S] */
    int32_t *recv_row;          /* [W(d)][W(s)][Tm][S] */
    int32_t *expert_num_tokens; /* [W][e_local] */
    int32_t *status;            /* [1] or NULL: cleared on the stream once the arguments
                                   are accepted, then set to the call's first device-side
                                   EP_ERR_* (bad id, repeated id, num_tokens out of range),
                                   if any. Left untouched when the call returns an error
                                   before that. */
} ep_route_outputs_t;

/*
 * ep_route_static -- the routing step of ep_dispatch (slot and row assignment,
 * counts, received-slot metadata) for callers that cannot allocate device
 * memory. The pages have no counterpart: it exists for this library's users.
 *
 * Who needs it: code whose device memory is owned by someone else and planned
 * up front -- an inference engine that reserves its memory pool at start-up,
 * or a plugin whose host framework forbids allocating after initialisation --
 * and code on a latency-critical path where a cudaMalloc (which may
 * synchronise the device) is not acceptable. Such callers cannot create the
 * workspace ep_ctx_create needs.
 *
 * It allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine. Its scratch is a static device array of EP_STATIC_SCRATCH_BYTES
 * (4 MiB) that every GPU loading this library holds until the process exits.
 * Problems needing more scratch than that -- roughly
 * W * ceil(max_tokens / 64) * ((W + E) * 8 + 128) bytes -- are refused with
 * EP_ERR_SCRATCH_LIMIT before anything is enqueued.
 *
 * The caller passes inputs (device: num_tokens or NULL, topk_ids, topk_weights,
 * as for ep_dispatch) and every output buffer (device, in *out). Results equal
 * the routing metadata ep_dispatch leaves in its workspace for the same inputs.
 *
 * The first call on each device also performs a one-time set-up (it looks up
 * the array's device address with that device current); make that first call
 * before any stream capture. All calls on a device share the one array, which
 * keeps the previous call's contents: each call clears what must start at
 * zero on its stream. Calls that overlap on the GPU (two streams, or two host
 * threads without ordering between their streams) race on the array.
 *
 * Every pointer (inputs, outputs, status) must be 4-byte aligned.
 *
 * Host-side errors: EP_ERR_INVALID_ARG (bad config, null or misaligned
 * pointer), EP_ERR_SCRATCH_LIMIT, EP_ERR_CUDA. Device-side errors go to
 * out->status.
 */
int ep_route_static(const ep_config_t *cfg, const int32_t *num_tokens, const int32_t *topk_ids,
                    const float *topk_weights, const ep_route_outputs_t *out, void *stream);

/*
 * Buffers of ep_agrs, all device memory owned by the caller.
 *   x_g    [W(d)][W*Tm][h] bf16  every rank's all-gathered token rows
 *   ids_g  [W(d)][W*Tm][K] int32 every rank's all-gathered top-k ids
 *   w_g    [W(d)][W*Tm][K] float every rank's all-gathered top-k weights
 *   y      [W(d)][W*Tm][h] bf16  each rank's expert output for every gathered token
 *   status [1] int32 or NULL     cleared at the start of the call, then set to the
 *                                first device-side EP_ERR_* (bad or repeated id,
 *                                num_tokens out of range) if any
 * Row (s*Tm + t) of a rank's block belongs to token t of rank s; rows of tokens
 * at or past num_tokens[s] are neither written nor read.
 */
typedef struct ep_agrs_buffers {
    void *x_g;
    int32_t *ids_g;
    float *w_g;
    void *y;
    int32_t *status;
} ep_agrs_buffers_t;

/*
 * ep_agrs -- the all-gather / reduce-scatter route of vLLM's AgRsAll2AllManager
 * (page device_communicators/all2all: its `dispatch` gathers every rank's
 * hidden states, top-k weights and top-k ids to every rank with all_gatherv;
 * its `combine` hands each rank back its own tokens with reduce_scatterv),
 * with identity experts between the two, for comparison with the all-to-all
 * route of ep_dispatch / ep_combine. It uses no context; three kernels run on
 * `stream`:
 *   1. all-gather: x_g[d][s*Tm+t] = a1[s][t] for every rank d, and the same for
 *      ids and weights, for each token t < num_tokens[s];
 *   2. experts, on each rank d (the fused-MoE step with an expert map): y[d][g]
 *      = bf16 of the fp32 fold, in top-k order, of w_k * x_g over the token's
 *      kept pairs whose expert lives on d (id / e_local == d), zero if none.
 *      Pairs are kept by ep_dispatch's rule: negative ids dropped, ids >= E
 *      and repeats of an id in a row dropped and reported;
 *   3. reduce-scatter: out[s][t] = the sum over d = 0..W-1, ascending, of
 *      y[d][s*Tm+t] in out_dtype (EP_BF16: each sum rounded to bf16; EP_F32:
 *      fp32 sums); zero for t >= num_tokens[s].
 * With identity experts the result equals ep_combine_two_stage after an
 * ep_dispatch of the same inputs, bit for bit: both sum one bf16 partial per
 * destination rank, ranks ascending.
 *
 * Inputs: num_tokens [W] int32 device or NULL (every rank holds max_tokens);
 * a1 [W][Tm][h] bf16, topk_ids and topk_weights [W][Tm][K] (device, as for
 * ep_dispatch); out [W][Tm][h] out_dtype (device). a1, x_g, y and out 16-byte
 * aligned. cfg->x_dtype must be EP_BF16; EP_FLAG_WEIGHT_ON_INPUT is refused;
 * the other flags and the extra payloads do not apply to this route and are
 * ignored. Sizes: W * W * max_tokens * hidden / 8 < 2^31; x_g and y take
 * 2 * W^2 * max_tokens * hidden bytes each -- W times the token bytes, which is
 * why the route suits small W.
 *
 * Host-side errors: EP_ERR_INVALID_ARG (bad config, dtype, flag, size, null or
 * misaligned pointer), EP_ERR_CUDA. Device-side errors go to buf->status.
 */
int ep_agrs(const ep_config_t *cfg, const int32_t *num_tokens, const void *a1,
            const int32_t *topk_ids, const float *topk_weights, const ep_agrs_buffers_t *buf,
            int32_t out_dtype, void *out, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* EP_H */
