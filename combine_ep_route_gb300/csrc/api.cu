// api.cu -- the C-ABI of the EP dispatch/combine library (declared in
// include/ep.h): configuration checks, workspace layout, the dispatch/combine
// state rule, kernel launches on the caller's stream, status readback and the
// per-kernel event timing used by the benchmark.
#include "ep_internal.cuh"

#include <nvtx3/nvToolsExt.h>

#include <cstddef>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

using ep::Layout;

namespace {

constexpr int kIdle = 0, kDispatched = 1;
constexpr int kCombineCtasPerSm = 3;   // default cap on the combine's resident CTAs per SM
constexpr int kCombineSmallKCtas = 16;  // default combine grid per SM for top_k up to 4
constexpr int kCombineFewRounds = 4;     // work items per thread of a full wave, at most, for
                                         // the combine to keep every CTA that fits

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bytes of one dispatched activation row: bf16 (2 per element), fp8 (1) or
// packed fp4 (two elements per byte). 0 for an unknown type.
long long x_row_bytes(const ep_config_t *c) {
    switch (c->x_dtype) {
        case EP_BF16: return 2LL * c->hidden;
        case EP_FP8: return (long long)c->hidden;
        case EP_FP4X2: return c->hidden % 2 ? 0 : c->hidden / 2;
        default: return 0;
    }
}

bool config_ok(const ep_config_t *c) {
    if (!c) return false;
    if (c->W < 1 || c->W > EP_MAX_W) return false;
    if (c->E < c->W || c->E > EP_MAX_E || c->E % c->W != 0) return false;
    if (c->top_k < 1 || c->top_k > EP_MAX_TOPK || c->top_k > c->E) return false;
    // hidden: the bf16 rows of expert_out and out need 2*h % 16 == 0; the
    // dispatched rows (bf16, fp8 or packed fp4) must be whole 16-byte vectors too
    if (c->max_tokens < 1 || c->hidden < 8 || (2LL * c->hidden) % 16 != 0) return false;
    const long long xb = x_row_bytes(c);
    if (xb <= 0 || xb % 16 != 0) return false;
    if (c->n_extra < 0 || c->n_extra > EP_MAX_EXTRA) return false;
    long long rb = xb;
    for (int i = 0; i < c->n_extra; ++i) {
        if (c->extra_row_bytes[i] <= 0 || c->extra_row_bytes[i] % 16 != 0) return false;
        rb += c->extra_row_bytes[i];
    }
    if (c->flags & ~(EP_FLAG_ZERO_PAD | EP_FLAG_SENDBUF | EP_FLAG_WEIGHT_ON_INPUT)) return false;
    // the page applies router weights on input for top_k == 1 only (and scales bf16 rows)
    if ((c->flags & EP_FLAG_WEIGHT_ON_INPUT) && (c->top_k != 1 || c->x_dtype != EP_BF16))
        return false;
    // a row must fit twice into one mover CTA's stage memory
    if (2 * align_up((size_t)rb, 128) > ep::kMoveSmemBudget) return false;
    // flat expert row indices (E * Ecap) and flat pair indices stay within int32
    const long long ecap = (long long)c->max_tokens * c->W;
    if ((long long)c->E * ecap >= (1LL << 31)) return false;
    if ((long long)c->W * c->W * c->max_tokens * c->top_k >= (1LL << 31)) return false;
    // combine work items (token, 16-byte vector) stay within 2^31
    if ((long long)c->W * c->max_tokens * (c->hidden / 8) >= (1LL << 31)) return false;
    return true;
}

void compute_layout(const ep_config_t *c, Layout *L) {
    const int W = c->W, Tm = c->max_tokens, K = c->top_k;
    L->e_local = c->E / W;
    L->S = K < L->e_local ? K : L->e_local;
    L->Ecap = Tm * W;
    L->tiles_per_rank = (Tm + ep::kRouteTile - 1) / ep::kRouteTile;
    L->num_tiles = W * L->tiles_per_rank;
    L->n_ctr = W + c->E;
    uint32_t rb = (uint32_t)x_row_bytes(c);
    for (int i = 0; i < c->n_extra; ++i) rb += (uint32_t)c->extra_row_bytes[i];
    L->row_bytes = rb;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, ep::kAlign);
        return at;
    };
    const size_t pairs = (size_t)W * Tm * K;
    const size_t slots = (size_t)W * W * Tm * L->S;
    L->hdr = take(sizeof(ep::DevHeader));
    L->tile_flag = take((size_t)L->num_tiles * ep::kFlagStride * 4);
    L->tile_agg = take((size_t)L->num_tiles * L->n_ctr * 4);
    L->tile_incl = take((size_t)L->num_tiles * L->n_ctr * 4);
    L->send_cnt = take((size_t)W * W * 4);
    L->pair_row = take(pairs * 4);
    L->pair_w = take(pairs * 4);
    L->pair_send = take(pairs * 4);
    L->recv_eloc = take(slots * 4);
    L->recv_w = take(slots * 4);
    L->recv_row = take(slots * 4);
    if (c->flags & EP_FLAG_SENDBUF) {
        L->send_x = take((size_t)W * W * Tm * rb);
        L->recv_x = take((size_t)W * W * Tm * rb);
    } else {
        L->send_x = L->recv_x = (size_t)-1;
    }
    L->total = off;
}

}  // namespace

struct ep_ctx {
    ep_config_t cfg;
    Layout L;
    uint8_t *ws;
    size_t ws_bytes;
    int state;
    bool initialized;
    int num_sms;
    // options
    uint64_t wait_limit_ns;
    int timing;
    int pdl;
    int move_ctas_per_sm;
    int move_pipes;
    int fault_skip;
    int combine_ctas_per_sm;
    int combine_wave[2];     // resident combine CTAs per SM (bf16, f32 out), 0 until queried
    int fused_dispatch;      // routing and row movement in one persistent launch
    int route_ctas;          // CTAs of that launch that route (0 = all, -1 = chosen per problem)
    int move_chunk_target;   // bytes; 0 = whole rows, -1 = chosen per problem
    int move_max_stages;     // -1 = chosen per problem (as move_pipes)
    int small_dispatch;      // small batches: the one-launch dispatch without waits (-1 auto, 0 off)
    // counters and event timing
    int64_t launches[EP_K_COUNT];
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pending[EP_K_COUNT];
    std::vector<cudaEvent_t> pool;
};

namespace {

template <class T>
T *ws_ptr(const ep_ctx *c, size_t off) {
    return reinterpret_cast<T *>(c->ws + off);
}

cudaEvent_t take_event(ep_ctx *c) {
    if (!c->pool.empty()) {
        cudaEvent_t e = c->pool.back();
        c->pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Records an event pair around one kernel launch when timing is on.
const char *const kKindRange[EP_K_COUNT] = {
    "ep:route", "ep:move_fused", "ep:pack", "ep:exchange", "ep:deliver",
    "ep:combine", "ep:zero_pad", "ep:combine_two_stage", "ep:dispatch_fused", "ep:dispatch_small"};

// Around every library launch: a launch count, an NVTX range named for the
// kernel (visible to Nsight tools; free when none is attached) and, with
// EP_OPT_KERNEL_TIMING, CUDA events on the launching stream.
struct KernelTimer {
    ep_ctx *c;
    int kind;
    cudaStream_t st;
    cudaEvent_t a = nullptr, b = nullptr;
    KernelTimer(ep_ctx *c_, int kind_, cudaStream_t st_) : c(c_), kind(kind_), st(st_) {
        nvtxRangePushA(kKindRange[kind]);
        c->launches[kind]++;
        if (c->timing) {
            a = take_event(c);
            b = take_event(c);
            if (a) cudaEventRecord(a, st);
        }
    }
    ~KernelTimer() {
        if (a && b) {
            cudaEventRecord(b, st);
            c->pending[kind].emplace_back(a, b);
        } else {
            if (a) c->pool.push_back(a);
            if (b) c->pool.push_back(b);
        }
        nvtxRangePop();
    }
};

int lazy_init(ep_ctx *c, cudaStream_t st) {
    if (c->initialized) return EP_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EP_ERR_CUDA;
    if (cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return EP_ERR_CUDA;
    // header and tile flags start at zero; the rest is written before it is read
    if (cudaMemsetAsync(c->ws, 0, c->L.tile_agg, st) != cudaSuccess) return EP_ERR_CUDA;
    c->initialized = true;
    return EP_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

void fill_move_common(const ep_ctx *c, ep::MoveParams &m) {
    const ep_config_t &cf = c->cfg;
    std::memset(&m, 0, sizeof(m));
    m.W = cf.W;
    m.K = cf.top_k;
    m.Tm = cf.max_tokens;
    m.S = c->L.S;
    m.e_local = c->L.e_local;
    m.Ecap = c->L.Ecap;
    m.n_seg = 1 + cf.n_extra;
    m.seg_bytes[0] = (uint32_t)x_row_bytes(&cf);
    m.seg_off[0] = 0;
    for (int i = 0; i < cf.n_extra; ++i) {
        m.seg_bytes[1 + i] = (uint32_t)cf.extra_row_bytes[i];
        m.seg_off[1 + i] = m.seg_off[i] + m.seg_bytes[i];
    }
    m.row_bytes = c->L.row_bytes;
    m.pair_row = ws_ptr<int32_t>(c, c->L.pair_row);
    m.pair_send = ws_ptr<int32_t>(c, c->L.pair_send);
    m.send_cnt = ws_ptr<int32_t>(c, c->L.send_cnt);
    m.recv_eloc = ws_ptr<int32_t>(c, c->L.recv_eloc);
    m.recv_row = ws_ptr<int32_t>(c, c->L.recv_row);
    if (cf.flags & EP_FLAG_SENDBUF) {
        m.send_x = ws_ptr<uint8_t>(c, c->L.send_x);
        m.recv_x = ws_ptr<uint8_t>(c, c->L.recv_x);
    }
    m.n_tokens = cf.W * cf.max_tokens;
    m.n_rows = cf.E * c->L.Ecap;
    m.n_slots = cf.W * cf.W * cf.max_tokens;
    m.hdr = ws_ptr<ep::DevHeader>(c, c->L.hdr);
    m.wait_limit_ns = c->wait_limit_ns;
}

// Pipelines per CTA, stages per pipeline and the dynamic shared memory of one
// mover CTA for the current options.
// Chunks per row: the largest count whose chunk is at least the target size
// and a multiple of 16 bytes that divides the activation row.
int move_chunks(const ep_ctx *c, int chunk_target) {
    const uint32_t a1b = (uint32_t)x_row_bytes(&c->cfg);
    if (chunk_target == 0) return 1;
    int best = 1;
    for (int n = 2; n <= 64; ++n) {
        if (a1b % (16u * n) != 0) continue;
        if (a1b / n < (uint32_t)chunk_target) break;
        best = n;
    }
    return best;
}

// The mover's unit size, pipelines per CTA and stages per pipeline: the
// options where set, else chosen per problem. Measured on GB300 (one-launch
// dispatch, prefill shape unless noted): small bulk copies (1 KiB, or 2 KiB
// on four pipelines) lose up to 2x; with top_k <= 2 a unit writes little, so
// larger units on four pipelines win (top_k 1: 57 us vs 78 us with the
// top_k-8 shape); rows of at most 4 KiB move best whole on eight pipelines of
// two stages (packed fp4 rows 80 vs 88 us, decode 24.1 vs 25.3 us); chunks of
// 3 KiB or more do better on four pipelines (fp8 rows 105 vs 115 us); bf16
// rows with top_k 8 are fastest in 2 KiB chunks, eight pipelines, four stages.
// The slot-sourced and send-buffer steps keep that last shape.
void move_options(const ep_ctx *c, int mode, int &chunk_target, int &pipes, int &max_stages) {
    chunk_target = 2048;
    pipes = 8;
    max_stages = 4;
    if (mode == ep::MOVE_FUSED) {
        const long long a1b = x_row_bytes(&c->cfg);
        if (c->cfg.top_k <= 2) {
            chunk_target = 4096;
            pipes = 4;
        } else if (a1b <= 4096) {
            chunk_target = 0;
            max_stages = 2;
        } else if (a1b / move_chunks(c, chunk_target) >= 3072) {
            pipes = 4;
        }
    }
    if (c->move_chunk_target >= 0) chunk_target = c->move_chunk_target;
    if (c->move_pipes > 0) pipes = c->move_pipes;
    if (c->move_max_stages > 0) max_stages = c->move_max_stages;
}

void move_shape(const ep_ctx *c, int chunks, int want_pipes, int max_stages, int &pipes, int &stages,
                uint32_t &stage_bytes, size_t &smem) {
    const uint32_t a1b = (uint32_t)x_row_bytes(&c->cfg);
    stage_bytes = (uint32_t)align_up(a1b / chunks + (c->L.row_bytes - a1b), 128);
    const int ctas = c->move_ctas_per_sm;
    size_t budget = ctas == 1 ? ep::kMoveSmemBudget : (size_t)(220 * 1024) / ctas - 2048;
    if (budget > ep::kMoveSmemBudget) budget = ep::kMoveSmemBudget;
    int total = (int)(budget / stage_bytes);
    pipes = want_pipes;
    while (pipes > 1 && total / pipes < 2) --pipes;
    stages = total / pipes;
    if (stages > max_stages) stages = max_stages;
    if (stages < 2) stages = 2;
    const int W = c->cfg.W;
    smem = (size_t)pipes * stages * stage_bytes + (size_t)pipes * stages * 8 +
           (size_t)pipes * stages * (ep::kMaxDst + 3) * 4 + (size_t)(W * W + 1) * 4;
}

// Mover parameters and launch shape for one mode.
void build_move(ep_ctx *c, int mode, const void *a1, const void *const *extra_in, void *b_a1,
                void *const *extra_out, ep::MoveParams &m, int &grid, int &block, size_t &smem_out) {
    fill_move_common(c, m);
    m.src_seg[0] = static_cast<const uint8_t *>(a1);
    m.dst_seg[0] = static_cast<uint8_t *>(b_a1);
    for (int i = 0; i < c->cfg.n_extra; ++i) {
        m.src_seg[1 + i] = static_cast<const uint8_t *>(extra_in[i]);
        m.dst_seg[1 + i] = static_cast<uint8_t *>(extra_out[i]);
    }
    // Token-sourced steps (fused, pack) have one unit per token: rows are split
    // into chunks so every pipeline gets many equal units. Slot-sourced steps
    // (exchange, deliver) have one unit per sent slot, already plentiful: whole
    // rows keep the bulk copies per byte low.
    int chunk_target, want_pipes, max_stages;
    move_options(c, mode, chunk_target, want_pipes, max_stages);
    const int chunks = (mode == ep::MOVE_FUSED || mode == ep::MOVE_PACK) ? move_chunks(c, chunk_target) : 1;
    int pipes, stages;
    uint32_t stage_bytes;
    size_t smem;
    move_shape(c, chunks, want_pipes, max_stages, pipes, stages, stage_bytes, smem);
    m.pipes = pipes;
    m.stages = stages;
    m.stage_bytes = stage_bytes;
    m.chunks = chunks;
    m.chunk_bytes = m.seg_bytes[0] / (uint32_t)m.chunks;
    grid = c->num_sms * c->move_ctas_per_sm;
    block = pipes * 32;
    smem_out = smem;
}

// Routers of the one-launch dispatch, when not set. Measured on GB300: with
// many tiles, 32 routers working through them in ticket order keep ahead of
// the movers while the other CTAs move rows from the outset (prefill: 174 us
// vs 179 us with every CTA routing first); with few tiles every CTA routes.
// The routers must publish tiles at least twice as fast as the movers consume
// them: a tile takes a router about 4 us + 0.75 us per top_k slot under load
// (10 us at top_k 8, from per-tile timestamps), and the movers drain a tile's
// rows (64 tokens, one read and top_k writes) at about 6.5 TB/s. Tiles of small
// rows therefore need more routers, up to every CTA (measured: packed fp4 rows
// 71 vs 80 us, 512-byte rows on 256 tiles 76 vs 112 us, against 32 routers).
int auto_route_ctas(const ep_ctx *c) {
    if (c->L.num_tiles <= 32) return 0;
    const double tile_bytes = (double)ep::kRouteTile * (1 + c->cfg.top_k) * (double)c->L.row_bytes;
    const double tile_time = (4.0 + 0.75 * c->cfg.top_k) * 1e-6;
    const double need = 2.0 * tile_time * 6.5e12 / tile_bytes;
    if (need >= (double)c->num_sms) return 0;
    return need > 32.0 ? (int)need + 1 : 32;
}

// Token slots per CTA of the small-batch dispatch (dispatch_small.cu), or 0
// when the batch does not qualify: its ids must be few enough for every CTA to
// read (W * max_tokens * top_k <= kSmallMaxIds), one CTA per SM must cover the
// slots with at most kSmallMaxTokens each, and their rows must fit in shared
// memory. Needs num_sms (set on first use).
int small_n_per(const ep_ctx *c, uint32_t *stage_bytes, size_t *smem, int *threads) {
    if (c->small_dispatch == 0 || c->num_sms < 1) return 0;
    const ep_config_t &cf = c->cfg;
    const long long slots = (long long)cf.W * cf.max_tokens;
    if (slots * cf.top_k > ep::kSmallMaxIds) return 0;
    const long long n_per = (slots + c->num_sms - 1) / c->num_sms;
    if (n_per > ep::kSmallMaxTokens) return 0;
    const uint32_t sb = (uint32_t)align_up(c->L.row_bytes, 128);
    // the most threads whose warp-private counters still fit
    int nt = ep::small_threads(cf.top_k);
    size_t bytes = ep::small_smem_bytes((int)n_per, sb, c->L.n_ctr, cf.top_k, cf.W, nt);
    while (bytes > ep::kMoveSmemBudget && nt > 256) {
        nt /= 2;
        bytes = ep::small_smem_bytes((int)n_per, sb, c->L.n_ctr, cf.top_k, cf.W, nt);
    }
    if (bytes > ep::kMoveSmemBudget) return 0;
    *stage_bytes = sb;
    *smem = bytes;
    *threads = nt;
    return (int)n_per;
}

int launch_move_mode(ep_ctx *c, int mode, int kind, const void *a1, const void *const *extra_in,
                     void *b_a1, void *const *extra_out, bool pdl, cudaStream_t st) {
    ep::MoveParams m;
    int grid, block;
    size_t smem;
    build_move(c, mode, a1, extra_in, b_a1, extra_out, m, grid, block, smem);
    KernelTimer tm(c, kind, st);
    return ep::launch_move(mode, m, grid, block, smem, pdl && !c->timing, st) == cudaSuccess
               ? EP_OK
               : EP_ERR_CUDA;
}

}  // namespace

extern "C" {

const char *ep_error_string(int code) {
    switch (code) {
        case EP_OK: return "ok";
        case EP_ERR_INVALID_ARG: return "invalid argument";
        case EP_ERR_CAPACITY: return "num_tokens outside [0, max_tokens]";
        case EP_ERR_STATE: return "dispatch/combine called out of order";
        case EP_ERR_EXPERT_ID: return "expert id >= num_experts (pair dropped)";
        case EP_ERR_DUPLICATE: return "expert id repeated within a token (later one dropped)";
        case EP_ERR_TIMEOUT: return "a bounded device wait expired";
        case EP_ERR_WORKSPACE: return "workspace too small or misaligned";
        case EP_ERR_CUDA: return "CUDA error";
        case EP_ERR_SCRATCH_LIMIT: return "problem too large for the static scratch of ep_route_static";
        default: return "unknown status";
    }
}

int ep_capacities(const ep_config_t *cfg, int32_t *tok_cap, int32_t *slots_per_token,
                  int32_t *expert_cap) {
    if (!config_ok(cfg) || !tok_cap || !slots_per_token || !expert_cap) return EP_ERR_INVALID_ARG;
    const int e_local = cfg->E / cfg->W;
    *tok_cap = cfg->max_tokens;
    *slots_per_token = cfg->top_k < e_local ? cfg->top_k : e_local;
    *expert_cap = cfg->max_tokens * cfg->W;
    return EP_OK;
}

int ep_workspace_bytes(const ep_config_t *cfg, size_t *bytes) {
    if (!config_ok(cfg) || !bytes) return EP_ERR_INVALID_ARG;
    Layout L;
    compute_layout(cfg, &L);
    *bytes = L.total;
    return EP_OK;
}

int ep_ctx_create(const ep_config_t *cfg, void *d_workspace, size_t workspace_bytes,
                  ep_ctx_t **out) {
    if (!config_ok(cfg) || !out) return EP_ERR_INVALID_ARG;
    *out = nullptr;
    if (!d_workspace) return EP_ERR_INVALID_ARG;
    Layout L;
    compute_layout(cfg, &L);
    if (workspace_bytes < L.total || !aligned(d_workspace, ep::kAlign)) return EP_ERR_WORKSPACE;
    ep_ctx *c = new (std::nothrow) ep_ctx();
    if (!c) return EP_ERR_INVALID_ARG;
    c->cfg = *cfg;
    c->L = L;
    c->ws = static_cast<uint8_t *>(d_workspace);
    c->ws_bytes = workspace_bytes;
    c->state = kIdle;
    c->initialized = false;
    c->num_sms = 0;
    c->wait_limit_ns = 2000000000ull;
    c->timing = 0;
    c->pdl = 0;   // measured: the step is faster without programmatic dependent launch
    c->move_ctas_per_sm = 1;
    c->move_pipes = -1;
    c->fault_skip = -1;
    c->combine_ctas_per_sm = 0;   // 0 = as many as fit (occupancy)
    c->combine_wave[0] = c->combine_wave[1] = 0;
    c->fused_dispatch = 1;
    c->route_ctas = -1;
    c->move_chunk_target = -1;
    c->move_max_stages = -1;
    c->small_dispatch = -1;
    for (int k = 0; k < EP_K_COUNT; ++k) c->launches[k] = 0;
    *out = c;
    return EP_OK;
}

int ep_ctx_destroy(ep_ctx_t *ctx) {
    if (!ctx) return EP_OK;
    for (int k = 0; k < EP_K_COUNT; ++k)
        for (auto &pr : ctx->pending[k]) {
            cudaEventDestroy(pr.first);
            cudaEventDestroy(pr.second);
        }
    for (cudaEvent_t e : ctx->pool) cudaEventDestroy(e);
    delete ctx;
    return EP_OK;
}

int ep_ctx_reset(ep_ctx_t *ctx) {
    if (!ctx) return EP_ERR_INVALID_ARG;
    ctx->state = kIdle;
    return EP_OK;
}

int ep_set_option(ep_ctx_t *ctx, int32_t option, int64_t value) {
    if (!ctx) return EP_ERR_INVALID_ARG;
    switch (option) {
        case EP_OPT_WAIT_LIMIT_NS:
            if (value < 1000 || value > 60000000000LL) return EP_ERR_INVALID_ARG;
            ctx->wait_limit_ns = (uint64_t)value;
            return EP_OK;
        case EP_OPT_KERNEL_TIMING:
            if (value != 0 && value != 1) return EP_ERR_INVALID_ARG;
            ctx->timing = (int)value;
            return EP_OK;
        case EP_OPT_PDL:
            if (value != 0 && value != 1) return EP_ERR_INVALID_ARG;
            ctx->pdl = (int)value;
            return EP_OK;
        case EP_OPT_MOVE_CTAS_PER_SM:
            if (value < 1 || value > 4) return EP_ERR_INVALID_ARG;
            ctx->move_ctas_per_sm = (int)value;
            return EP_OK;
        case EP_OPT_MOVE_PIPES:
            if (value != -1 && (value < 1 || value > 8)) return EP_ERR_INVALID_ARG;
            ctx->move_pipes = (int)value;
            return EP_OK;
        case EP_OPT_FAULT_SKIP_PUBLISH:
            if (value < -1 || value >= ctx->L.num_tiles) return EP_ERR_INVALID_ARG;
            ctx->fault_skip = (int)value;
            return EP_OK;
        case EP_OPT_COMBINE_CTAS_PER_SM:
            if (value < 0 || value > 16) return EP_ERR_INVALID_ARG;
            ctx->combine_ctas_per_sm = (int)value;
            return EP_OK;
        case EP_OPT_MOVE_CHUNK_BYTES:
            if (value != -1 && (value < 0 || value > (1 << 20) || value % 16 != 0)) return EP_ERR_INVALID_ARG;
            ctx->move_chunk_target = (int)value;
            return EP_OK;
        case EP_OPT_MOVE_MAX_STAGES:
            if (value != -1 && (value < 2 || value > 32)) return EP_ERR_INVALID_ARG;
            ctx->move_max_stages = (int)value;
            return EP_OK;
        case EP_OPT_FUSED_DISPATCH:
            if (value != 0 && value != 1) return EP_ERR_INVALID_ARG;
            ctx->fused_dispatch = (int)value;
            return EP_OK;
        case EP_OPT_ROUTE_CTAS:
            if (value < -1 || value > 4096) return EP_ERR_INVALID_ARG;
            ctx->route_ctas = (int)value;
            return EP_OK;
        case EP_OPT_SMALL_DISPATCH:
            if (value < -1 || value > 1) return EP_ERR_INVALID_ARG;
            ctx->small_dispatch = (int)value;
            return EP_OK;
        default: return EP_ERR_INVALID_ARG;
    }
}

int ep_get_metadata(const ep_ctx_t *ctx, ep_metadata_t *out) {
    if (!ctx || !out) return EP_ERR_INVALID_ARG;
    out->send_cnt = ws_ptr<int32_t>(ctx, ctx->L.send_cnt);
    out->pair_row = ws_ptr<int32_t>(ctx, ctx->L.pair_row);
    out->pair_w = ws_ptr<float>(ctx, ctx->L.pair_w);
    out->pair_send = ws_ptr<int32_t>(ctx, ctx->L.pair_send);
    out->recv_eloc = ws_ptr<int32_t>(ctx, ctx->L.recv_eloc);
    out->recv_w = ws_ptr<float>(ctx, ctx->L.recv_w);
    out->recv_row = ws_ptr<int32_t>(ctx, ctx->L.recv_row);
    const bool sb = ctx->cfg.flags & EP_FLAG_SENDBUF;
    out->send_x = sb ? ws_ptr<void>(ctx, ctx->L.send_x) : nullptr;
    out->recv_x = sb ? ws_ptr<void>(ctx, ctx->L.recv_x) : nullptr;
    out->slots_per_token = ctx->L.S;
    out->expert_cap = ctx->L.Ecap;
    out->row_bytes = (int32_t)ctx->L.row_bytes;
    out->reserved = 0;
    return EP_OK;
}

int ep_dispatch(ep_ctx_t *ctx, const void *a1, const int32_t *num_tokens, const int32_t *topk_ids,
                const float *topk_weights, const void *const *extra_in, void *b_a1,
                void *const *extra_out, int32_t *expert_num_tokens, int32_t path, void *stream) {
    if (!ctx || !a1 || !topk_ids || !topk_weights || !b_a1 || !expert_num_tokens)
        return EP_ERR_INVALID_ARG;
    const ep_config_t &cf = ctx->cfg;
    if (path != EP_PATH_FUSED && path != EP_PATH_SENDBUF) return EP_ERR_INVALID_ARG;
    if (path == EP_PATH_SENDBUF && !(cf.flags & EP_FLAG_SENDBUF)) return EP_ERR_WORKSPACE;
    if (!aligned(a1, 16) || !aligned(b_a1, 16) || !aligned(topk_ids, 4) ||
        !aligned(topk_weights, 4) || !aligned(expert_num_tokens, 4) ||
        (num_tokens && !aligned(num_tokens, 4)))
        return EP_ERR_INVALID_ARG;
    if (cf.n_extra > 0) {
        if (!extra_in || !extra_out) return EP_ERR_INVALID_ARG;
        for (int i = 0; i < cf.n_extra; ++i)
            if (!extra_in[i] || !extra_out[i] || !aligned(extra_in[i], 16) || !aligned(extra_out[i], 16))
                return EP_ERR_INVALID_ARG;
    }
    if (ctx->state != kIdle) return EP_ERR_STATE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int rc = lazy_init(ctx, st);
    if (rc != EP_OK) return rc;

    const Layout &L = ctx->L;
    ep::RouteParams rp;
    std::memset(&rp, 0, sizeof(rp));
    rp.ids = topk_ids;
    rp.weights = topk_weights;
    rp.num_tokens = num_tokens;
    rp.W = cf.W;
    rp.E = cf.E;
    rp.K = cf.top_k;
    rp.Tm = cf.max_tokens;
    rp.e_local = L.e_local;
    rp.S = L.S;
    rp.Ecap = L.Ecap;
    rp.tiles_per_rank = L.tiles_per_rank;
    rp.num_tiles = L.num_tiles;
    rp.n_ctr = L.n_ctr;
    rp.hdr = ws_ptr<ep::DevHeader>(ctx, L.hdr);
    rp.tile_flag = ws_ptr<uint32_t>(ctx, L.tile_flag);
    rp.tile_agg = ws_ptr<int32_t>(ctx, L.tile_agg);
    rp.tile_incl = ws_ptr<int32_t>(ctx, L.tile_incl);
    rp.send_cnt = ws_ptr<int32_t>(ctx, L.send_cnt);
    rp.pair_row = ws_ptr<int32_t>(ctx, L.pair_row);
    rp.pair_w = ws_ptr<float>(ctx, L.pair_w);
    rp.pair_send = ws_ptr<int32_t>(ctx, L.pair_send);
    rp.recv_eloc = ws_ptr<int32_t>(ctx, L.recv_eloc);
    rp.recv_w = ws_ptr<float>(ctx, L.recv_w);
    rp.recv_row = ws_ptr<int32_t>(ctx, L.recv_row);
    rp.expert_num_tokens = expert_num_tokens;
    rp.wait_limit_ns = ctx->wait_limit_ns;
    rp.fault_skip_tile = ctx->fault_skip;
    rp.vec_ids = aligned(topk_ids, 16) && aligned(topk_weights, 16);
    rp.vec_recv = L.S % 4 == 0;   // workspace regions are 256-byte aligned
    rp.unit_weights = (cf.flags & EP_FLAG_WEIGHT_ON_INPUT) ? 1 : 0;
    const bool pdl = ctx->pdl != 0;
    bool one_launch = ctx->fused_dispatch && path == EP_PATH_FUSED &&
                      !(cf.flags & EP_FLAG_WEIGHT_ON_INPUT);
    ep::MoveParams fm;
    int fgrid = 0, fblock = 0;
    size_t fsmem = 0;
    if (one_launch) {
        // routing and row movement in one persistent launch: one CTA per SM of the
        // routing step's 256 threads, of which the first move_pipes warps (at most
        // eight) run pipelines
        const int saved_ctas = ctx->move_ctas_per_sm;
        ctx->move_ctas_per_sm = 1;
        build_move(ctx, ep::MOVE_FUSED, a1, extra_in, b_a1, extra_out, fm, fgrid, fblock, fsmem);
        ctx->move_ctas_per_sm = saved_ctas;
        one_launch = fblock <= ep::kRouteThreads;
    }
    uint32_t small_sb = 0;
    size_t small_smem = 0;
    int small_nt = 0;
    const int small = one_launch ? small_n_per(ctx, &small_sb, &small_smem, &small_nt) : 0;
    if (small > 0) {
        ep::SmallParams sp;
        std::memset(&sp, 0, sizeof(sp));
        sp.rp = rp;
        fill_move_common(ctx, sp.mp);
        sp.mp.src_seg[0] = static_cast<const uint8_t *>(a1);
        sp.mp.dst_seg[0] = static_cast<uint8_t *>(b_a1);
        for (int i = 0; i < cf.n_extra; ++i) {
            sp.mp.src_seg[1 + i] = static_cast<const uint8_t *>(extra_in[i]);
            sp.mp.dst_seg[1 + i] = static_cast<uint8_t *>(extra_out[i]);
        }
        sp.n_per = small;
        sp.stage_bytes = small_sb;
        sp.div_tm = ep::make_fastdiv((uint32_t)cf.max_tokens);
        sp.div_el = ep::make_fastdiv((uint32_t)L.e_local);
        const int slots = cf.W * cf.max_tokens;
        const int grid = (slots + small - 1) / small;
        KernelTimer tm(ctx, EP_K_DISPATCH_SMALL, st);
        if (ep::launch_dispatch_small(sp, grid, small_nt, small_smem, st) != cudaSuccess)
            return EP_ERR_CUDA;
    } else if (one_launch) {
        fm.wait_tiles = 1;
        fm.dynamic_units = 1;
        fm.tile_flag = rp.tile_flag;
        fm.tiles_per_rank = L.tiles_per_rank;
        fm.div_tm = ep::make_fastdiv((uint32_t)cf.max_tokens);
        rp.route_ctas = ctx->route_ctas >= 0 ? ctx->route_ctas : auto_route_ctas(ctx);
        KernelTimer tm(ctx, EP_K_DISPATCH_FUSED, st);
        if (ep::launch_dispatch_fused(rp, fm, ctx->num_sms, fsmem, st) != cudaSuccess) return EP_ERR_CUDA;
    } else {
        KernelTimer tm(ctx, EP_K_ROUTE, st);
        if (ep::launch_route(rp, st) != cudaSuccess) return EP_ERR_CUDA;
    }
    if (one_launch) {
        // rows already moved
    } else if (cf.flags & EP_FLAG_WEIGHT_ON_INPUT) {
        // rows are scaled while they move: one register-path kernel to the b_a1
        // row (fused) or to the send row (send-buffer path, then the mover)
        ep::ScaleMoveParams sp;
        std::memset(&sp, 0, sizeof(sp));
        const bool fused = path == EP_PATH_FUSED;
        sp.a1 = static_cast<const uint8_t *>(a1);
        sp.weights = topk_weights;
        sp.dst_index = ws_ptr<int32_t>(ctx, fused ? L.pair_row : L.pair_send);
        sp.n_dst_rows = fused ? cf.E * L.Ecap : cf.W * cf.W * cf.max_tokens;
        sp.a1_bytes = 2u * (uint32_t)cf.hidden;
        sp.nvec_a1 = sp.a1_bytes / 16;
        sp.n_seg = 1 + cf.n_extra;
        sp.combined = fused ? 0 : 1;
        sp.vecs = sp.nvec_a1;
        sp.dst[0] = fused ? static_cast<uint8_t *>(b_a1) : ws_ptr<uint8_t>(ctx, L.send_x);
        sp.dst_stride[0] = fused ? sp.a1_bytes : L.row_bytes;
        uint32_t off = sp.a1_bytes;
        for (int i = 0; i < cf.n_extra; ++i) {
            sp.src_seg[1 + i] = static_cast<const uint8_t *>(extra_in[i]);
            sp.seg_vecs[1 + i] = (uint32_t)cf.extra_row_bytes[i] / 16;
            sp.seg_off[1 + i] = off;
            off += (uint32_t)cf.extra_row_bytes[i];
            sp.dst[1 + i] = fused ? static_cast<uint8_t *>(extra_out[i]) : nullptr;
            sp.dst_stride[1 + i] = (size_t)cf.extra_row_bytes[i];
            sp.vecs += sp.seg_vecs[1 + i];
        }
        const long long items = (long long)cf.W * cf.max_tokens * sp.vecs;
        if (items >= (1LL << 31)) return EP_ERR_INVALID_ARG;
        sp.n_items = (uint32_t)items;
        sp.div_vecs = ep::make_fastdiv(sp.vecs);
        {
            KernelTimer tm(ctx, fused ? EP_K_MOVE_FUSED : EP_K_PACK, st);
            if (ep::launch_scale_move(sp, ctx->num_sms * 8, st) != cudaSuccess) return EP_ERR_CUDA;
        }
        if (!fused) {
            rc = launch_move_mode(ctx, ep::MOVE_EXCHANGE, EP_K_EXCHANGE, a1, extra_in, b_a1, extra_out,
                                  pdl, st);
            if (rc == EP_OK)
                rc = launch_move_mode(ctx, ep::MOVE_DELIVER, EP_K_DELIVER, a1, extra_in, b_a1,
                                      extra_out, pdl, st);
            if (rc != EP_OK) return rc;
        }
    } else if (path == EP_PATH_FUSED) {
        rc = launch_move_mode(ctx, ep::MOVE_FUSED, EP_K_MOVE_FUSED, a1, extra_in, b_a1, extra_out, pdl, st);
        if (rc != EP_OK) return rc;
    } else {
        rc = launch_move_mode(ctx, ep::MOVE_PACK, EP_K_PACK, a1, extra_in, b_a1, extra_out, pdl, st);
        if (rc == EP_OK)
            rc = launch_move_mode(ctx, ep::MOVE_EXCHANGE, EP_K_EXCHANGE, a1, extra_in, b_a1, extra_out,
                                  pdl, st);
        if (rc == EP_OK)
            rc = launch_move_mode(ctx, ep::MOVE_DELIVER, EP_K_DELIVER, a1, extra_in, b_a1, extra_out,
                                  pdl, st);
        if (rc != EP_OK) return rc;
    }
    if (cf.flags & EP_FLAG_ZERO_PAD) {
        ep::ZeroPadParams zp;
        std::memset(&zp, 0, sizeof(zp));
        zp.n_seg = 1 + cf.n_extra;
        zp.seg_bytes[0] = (uint32_t)x_row_bytes(&cf);
        zp.dst_seg[0] = static_cast<uint8_t *>(b_a1);
        for (int i = 0; i < cf.n_extra; ++i) {
            zp.seg_bytes[1 + i] = (uint32_t)cf.extra_row_bytes[i];
            zp.dst_seg[1 + i] = static_cast<uint8_t *>(extra_out[i]);
        }
        zp.expert_num_tokens = expert_num_tokens;
        zp.E = cf.E;
        zp.Ecap = L.Ecap;
        zp.send_cnt = ws_ptr<int32_t>(ctx, L.send_cnt);
        zp.recv_eloc = ws_ptr<int32_t>(ctx, L.recv_eloc);
        zp.recv_w = ws_ptr<float>(ctx, L.recv_w);
        zp.recv_row = ws_ptr<int32_t>(ctx, L.recv_row);
        zp.W = cf.W;
        zp.Tm = cf.max_tokens;
        zp.S = L.S;
        KernelTimer tm(ctx, EP_K_ZERO_PAD, st);
        if (ep::launch_zero_pad(zp, 32, st) != cudaSuccess) return EP_ERR_CUDA;
    }
    ctx->state = kDispatched;
    return EP_OK;
}

int ep_combine(ep_ctx_t *ctx, const void *expert_out, int32_t out_dtype, void *out, void *stream) {
    if (!ctx || !expert_out || !out) return EP_ERR_INVALID_ARG;
    if (out_dtype != EP_BF16 && out_dtype != EP_F32) return EP_ERR_INVALID_ARG;
    if (!aligned(expert_out, 16) || !aligned(out, 16)) return EP_ERR_INVALID_ARG;
    if (ctx->state != kDispatched) return EP_ERR_STATE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const ep_config_t &cf = ctx->cfg;
    ep::CombineParams cp;
    cp.expert_out = static_cast<const uint8_t *>(expert_out);
    cp.pair_row = ws_ptr<int32_t>(ctx, ctx->L.pair_row);
    cp.pair_w = ws_ptr<float>(ctx, ctx->L.pair_w);
    cp.out = out;
    cp.K = cf.top_k;
    cp.h = cf.hidden;
    cp.n_tokens = cf.W * cf.max_tokens;
    cp.nvec = cf.hidden / 8;
    cp.n_rows = cf.E * ctx->L.Ecap;
    const int vpt = ep::combine_vectors_per_thread(cf.top_k);
    cp.groups = (cp.nvec + vpt - 1) / vpt;
    cp.div_groups = ep::make_fastdiv((uint32_t)cp.groups);
    const long long total = (long long)cp.n_tokens * cp.groups;
    long long grid = (total + 255) / 256;
    int per_sm = ctx->combine_ctas_per_sm;
    if (per_sm == 0 && cf.top_k <= 4) {
        // Small top_k: a grid of several waves. A thread reduces 2-4 vectors of its
        // token, and smaller CTAs taken up as others finish balance the end better:
        // measured on GB300 on the prefill shape, top_k 1 combine 42.8 -> 39.6 us,
        // top_k 2 60.2 -> 57.9 us, top_k 4 93.0 -> 92.6 us (8 per SM is close; at
        // top_k 8 the same grid is 1.5-3 % slower than one wave).
        per_sm = kCombineSmallKCtas;
    } else if (per_sm == 0) {
        int &cached = ctx->combine_wave[out_dtype == EP_F32 ? 1 : 0];
        if (cached == 0 && ep::combine_occupancy(cf.top_k, out_dtype == EP_F32, &cached) != cudaSuccess)
            return EP_ERR_CUDA;
        // At most three CTAs per SM, though four fit at top_k 8: measured on GB300,
        // fewer loads in flight make the prefill combine faster (169.3 -> 164.9 us; the
        // Zipf and grouped workloads 0.4 and 1.2 % faster; two per SM is 8-14 % slower).
        // A small batch, whose work items are done in a few rounds, keeps every CTA
        // that fits instead: one wave of four per SM took the decode step (1024
        // tokens, about two items per thread) from 21.3 to 20.7 us.
        const long long wave = (long long)ctx->num_sms * cached * 256;
        per_sm = total <= kCombineFewRounds * wave ? cached
                 : (cached < kCombineCtasPerSm ? cached : kCombineCtasPerSm);
    }
    const long long cap = (long long)ctx->num_sms * per_sm;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    {
        KernelTimer tm(ctx, EP_K_COMBINE, st);
        if (ep::launch_combine(cp, out_dtype == EP_F32, (int)grid, ctx->pdl && !ctx->timing, st) !=
            cudaSuccess)
            return EP_ERR_CUDA;
    }
    ctx->state = kIdle;
    return EP_OK;
}

int ep_combine_two_stage(ep_ctx_t *ctx, const void *expert_out, int32_t out_dtype, void *out,
                         void *stream) {
    if (!ctx || !expert_out || !out) return EP_ERR_INVALID_ARG;
    if (out_dtype != EP_BF16 && out_dtype != EP_F32) return EP_ERR_INVALID_ARG;
    if (!aligned(expert_out, 16) || !aligned(out, 16)) return EP_ERR_INVALID_ARG;
    if (!(ctx->cfg.flags & EP_FLAG_SENDBUF)) return EP_ERR_WORKSPACE;
    if (ctx->state != kDispatched) return EP_ERR_STATE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const ep_config_t &cf = ctx->cfg;
    const Layout &L = ctx->L;
    ep::PartialParams a;
    a.expert_out = static_cast<const uint8_t *>(expert_out);
    a.send_cnt = ws_ptr<int32_t>(ctx, L.send_cnt);
    a.recv_eloc = ws_ptr<int32_t>(ctx, L.recv_eloc);
    a.recv_row = ws_ptr<int32_t>(ctx, L.recv_row);
    a.recv_w = ws_ptr<float>(ctx, L.recv_w);
    a.part = ws_ptr<uint8_t>(ctx, L.recv_x);
    a.part_stride = L.row_bytes;
    a.W = cf.W;
    a.Tm = cf.max_tokens;
    a.S = L.S;
    a.e_local = L.e_local;
    a.Ecap = L.Ecap;
    a.h = cf.hidden;
    a.nvec = cf.hidden / 8;
    a.n_items = (uint32_t)((long long)cf.W * cf.W * cf.max_tokens * a.nvec);
    a.div_nvec = ep::make_fastdiv((uint32_t)a.nvec);
    a.div_tm = ep::make_fastdiv((uint32_t)cf.max_tokens);
    a.div_w = ep::make_fastdiv((uint32_t)cf.W);
    if ((long long)cf.W * cf.W * cf.max_tokens * a.nvec >= (1LL << 31)) return EP_ERR_INVALID_ARG;
    ep::GatherParams b;
    b.part = a.part;
    b.part_stride = a.part_stride;
    b.pair_send = ws_ptr<int32_t>(ctx, L.pair_send);
    b.out = out;
    b.W = cf.W;
    b.Tm = cf.max_tokens;
    b.K = cf.top_k;
    b.h = cf.hidden;
    b.nvec = a.nvec;
    b.n_items = (uint32_t)(cf.W * cf.max_tokens) * (uint32_t)b.nvec;
    b.div_nvec = a.div_nvec;
    b.div_tm = a.div_tm;
    {
        KernelTimer tm(ctx, EP_K_COMBINE_TWO_STAGE, st);
        if (ep::launch_combine_two_stage(a, b, out_dtype == EP_F32, ctx->num_sms, st) != cudaSuccess)
            return EP_ERR_CUDA;
        ctx->launches[EP_K_COMBINE_TWO_STAGE]++;   // two kernels under one timer
    }
    ctx->state = kIdle;
    return EP_OK;
}

int ep_status(ep_ctx_t *ctx, void *stream) {
    if (!ctx) return EP_ERR_INVALID_ARG;
    if (!ctx->initialized) return EP_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return EP_ERR_CUDA;
    ep::DevHeader h;
    if (cudaMemcpy(&h, ctx->ws + ctx->L.hdr, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
        return EP_ERR_CUDA;
    if (h.err != 0 || h.err_count != 0 || h.ticket != 0 || h.done != 0) {
        // clear the error words and counters; the epoch must survive (the tile
        // flags in the workspace carry earlier epochs)
        if (cudaMemset(ctx->ws + ctx->L.hdr, 0, offsetof(ep::DevHeader, epoch)) != cudaSuccess)
            return EP_ERR_CUDA;
    }
    if (h.err != 0) return h.err;
    if (h.ticket != 0 || h.done != 0) return EP_ERR_STATE;
    return EP_OK;
}

int ep_kernel_times(ep_ctx_t *ctx, ep_kernel_times_t *out) {
    if (!ctx || !out) return EP_ERR_INVALID_ARG;
    int rc = EP_OK;
    for (int k = 0; k < EP_K_COUNT; ++k) {
        out->launches[k] = ctx->launches[k];
        ctx->launches[k] = 0;
        double tot = 0.0;
        int64_t n = 0;
        for (auto &pr : ctx->pending[k]) {
            float ms = 0.f;
            if (cudaEventSynchronize(pr.second) == cudaSuccess &&
                cudaEventElapsedTime(&ms, pr.first, pr.second) == cudaSuccess) {
                tot += ms;
                ++n;
            } else {
                rc = EP_ERR_CUDA;
            }
            ctx->pool.push_back(pr.first);
            ctx->pool.push_back(pr.second);
        }
        ctx->pending[k].clear();
        out->total_ms[k] = tot;
        out->timed[k] = n;
    }
    return rc;
}

}  // extern "C"
