// agrs.cu -- ep_agrs: the all-gather / reduce-scatter route of vLLM's
// AgRsAll2AllManager (page device_communicators/all2all, `dispatch` and
// `combine`), with all W ranks simulated as blocks of one GPU's memory and the
// experts between the two collectives being the identity.
//
// Three kernels, one per step of the route:
//   gather  -- all_gatherv of hidden states, top-k ids and top-k weights: every
//              valid token row is read once and written into each rank's
//              gathered block (16-byte vectors for the rows, 4-byte words for
//              the ids and weights).
//   experts -- the fused-MoE step on each rank d with its expert map: for each
//              gathered token, the fp32 fold in top-k order of w_k * x over the
//              token's kept pairs whose expert lives on d, rounded to bf16.
//              One warp per (rank, token) row: lanes < K classify the pairs
//              once (negative ids dropped, ids >= E and repeats flagged and
//              dropped, the first occurrence kept), then every lane streams
//              16-byte vectors of the row. A row with no local pair is written
//              as zeros without reading x.
//   reduce  -- reduce_scatterv: out[s][t] = the sum over ranks d = 0..W-1,
//              ascending, of rank d's expert output for that token, in the
//              output type (bf16: each sum rounded; f32: fp32 sums). One thread
//              per 16-byte vector of bf16 input, up to 8 rank loads in flight.
// All three run as one-wave grid-stride grids. Products and sums are
// __fmul_rn / __fadd_rn, never contracted into an FMA.
#include "ep_internal.cuh"

#include <cuda_bf16.h>
#include <nvtx3/nvToolsExt.h>

#include <mutex>

namespace {

using ep::FastDiv;
using ep::fastdiv;
using ep::make_fastdiv;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxDevices = 64;

struct AgrsParams {
    const uint8_t *a1;            // [W][Tm][h] bf16
    const int32_t *ids;           // [W][Tm][K]
    const float *weights;         // [W][Tm][K]
    const int32_t *num_tokens;    // [W] or null
    uint8_t *x_g;                 // [W(d)][W*Tm][h] bf16
    int32_t *ids_g;               // [W(d)][W*Tm][K]
    float *w_g;                   // [W(d)][W*Tm][K]
    uint8_t *y;                   // [W(d)][W*Tm][h] bf16
    void *out;                    // [W][Tm][h] bf16 or f32
    int32_t *status;              // [1] or null
    int W, E, K, Tm, e_local, h, nvec;
    uint32_t n_tok;               // W * Tm gathered rows per rank
    FastDiv div_nvec, div_K, div_Tm, div_ntok;
};

__device__ __forceinline__ void report(int32_t *status, int32_t code) {
    if (status) atomicCAS(status, 0, code);
}

// Tokens rank s holds (num_tokens clamped to [0, Tm]; Tm without a count).
__device__ __forceinline__ int held(const AgrsParams &p, int s) {
    if (!p.num_tokens) return p.Tm;
    const int n = __ldg(p.num_tokens + s);
    return n < 0 ? 0 : (n > p.Tm ? p.Tm : n);
}

__device__ __forceinline__ uint4 ld_stream_v4(const void *ptr) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr));
    return v;
}

__device__ __forceinline__ void fold2(float &a0, float &a1, float w, uint32_t x) {
    a0 = __fadd_rn(a0, __fmul_rn(w, __uint_as_float(x << 16)));
    a1 = __fadd_rn(a1, __fmul_rn(w, __uint_as_float(x & 0xFFFF0000u)));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_round(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}

// ----------------------------------------------------------------- all-gather
__global__ void __launch_bounds__(kThreads) agrs_gather_kernel(const AgrsParams p) {
    if (blockIdx.x == 0 && (int)threadIdx.x < p.W && p.num_tokens) {
        const int n = p.num_tokens[threadIdx.x];
        if (n < 0 || n > p.Tm) report(p.status, EP_ERR_CAPACITY);
    }
    const size_t row_bytes = (size_t)p.h * 2;
    const size_t plane_x = (size_t)p.n_tok * row_bytes;       // one rank's gathered rows
    const size_t plane_k = (size_t)p.n_tok * p.K;             // one rank's gathered ids
    const uint32_t nx = p.n_tok * (uint32_t)p.nvec;
    const uint32_t total = nx + (uint32_t)plane_k;            // < 2^31 (checked on the host)
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        if (i < nx) {
            const uint32_t g = fastdiv(i, p.div_nvec);
            const uint32_t v = i - g * (uint32_t)p.nvec;
            const uint32_t s = fastdiv(g, p.div_Tm);
            if ((int)(g - s * (uint32_t)p.Tm) >= held(p, (int)s)) continue;
            const size_t off = (size_t)g * row_bytes + (size_t)v * 16;
            const uint4 x = ld_stream_v4(p.a1 + off);
            uint8_t *dst = p.x_g + off;
            for (int d = 0; d < p.W; ++d, dst += plane_x) *reinterpret_cast<uint4 *>(dst) = x;
        } else {
            const uint32_t j = i - nx;
            const uint32_t g = fastdiv(j, p.div_K);
            const uint32_t s = fastdiv(g, p.div_Tm);
            if ((int)(g - s * (uint32_t)p.Tm) >= held(p, (int)s)) continue;
            const int32_t id = __ldg(p.ids + j);
            const float w = __ldg(p.weights + j);
            for (int d = 0; d < p.W; ++d) {
                p.ids_g[(size_t)d * plane_k + j] = id;
                p.w_g[(size_t)d * plane_k + j] = w;
            }
        }
    }
}

// -------------------------------------------------------- experts on each rank
__global__ void __launch_bounds__(kThreads) agrs_experts_kernel(const AgrsParams p) {
    __shared__ float sw[kWarps][EP_MAX_TOPK];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const size_t row_bytes = (size_t)p.h * 2;
    const uint32_t rows = (uint32_t)p.W * p.n_tok;            // (rank, gathered token)
    for (uint32_t r = blockIdx.x * kWarps + wib; r < rows; r += gridDim.x * kWarps) {
        const uint32_t d = fastdiv(r, p.div_ntok);
        const uint32_t g = r - d * p.n_tok;
        const uint32_t s = fastdiv(g, p.div_Tm);
        if ((int)(g - s * (uint32_t)p.Tm) >= held(p, (int)s)) continue;   // warp-uniform
        // classify the token's pairs from rank d's gathered copy
        const size_t kb = (size_t)r * p.K;                    // == d*plane_k + g*K
        int32_t e = -1;
        float w = 0.f;
        if (lane < p.K) {
            e = p.ids_g[kb + lane];
            w = p.w_g[kb + lane];
        }
        const bool in_range = lane < p.K && e >= 0 && e < p.E;
        if (d == 0 && lane < p.K && e >= p.E) report(p.status, EP_ERR_EXPERT_ID);
        // lanes out of range get a key no other lane has
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, in_range ? e : -1 - lane);
        const bool kept = in_range && (__ffs(peers) - 1 == lane);
        if (d == 0 && in_range && !kept) report(p.status, EP_ERR_DUPLICATE);
        const bool local = kept && (uint32_t)(e / p.e_local) == d;
        const uint32_t mask = __ballot_sync(0xFFFFFFFFu, local);
        if (lane < p.K) sw[wib][lane] = w;
        __syncwarp();
        const uint8_t *xrow = p.x_g + (size_t)r * row_bytes;
        uint8_t *yrow = p.y + (size_t)r * row_bytes;
        if (mask == 0) {
            for (int v = lane; v < p.nvec; v += 32)
                *reinterpret_cast<uint4 *>(yrow + (size_t)v * 16) = make_uint4(0u, 0u, 0u, 0u);
        } else {
            // eight 16-byte loads per lane in flight before the fold (measured on
            // GB300, the route's whole step: prefill 626 -> 623 us, Zipf 620 ->
            // 615 us against four; 73 registers, three CTAs per SM instead of
            // four; prefetching the next row's ids and weights as well gained
            // nothing more)
            for (int v0 = lane; v0 < p.nvec; v0 += 8 * 32) {
                uint4 x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int v = v0 + u * 32;
                    x[u] = v < p.nvec ? ld_stream_v4(xrow + (size_t)v * 16) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int v = v0 + u * 32;
                    if (v >= p.nvec) break;
                    float a[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) a[i] = 0.f;
                    for (uint32_t m = mask; m; m &= m - 1) {
                        const float wk = sw[wib][__ffs(m) - 1];
                        fold2(a[0], a[1], wk, x[u].x);
                        fold2(a[2], a[3], wk, x[u].y);
                        fold2(a[4], a[5], wk, x[u].z);
                        fold2(a[6], a[7], wk, x[u].w);
                    }
                    uint4 o;
                    o.x = pack_bf16x2(a[0], a[1]);
                    o.y = pack_bf16x2(a[2], a[3]);
                    o.z = pack_bf16x2(a[4], a[5]);
                    o.w = pack_bf16x2(a[6], a[7]);
                    *reinterpret_cast<uint4 *>(yrow + (size_t)v * 16) = o;
                }
            }
        }
        __syncwarp();   // sw is rewritten by this warp's next row
    }
}

// ------------------------------------------------------------- reduce-scatter
template <bool OUT_F32>
__global__ void __launch_bounds__(kThreads) agrs_reduce_kernel(const AgrsParams p) {
    const size_t row_bytes = (size_t)p.h * 2;
    const size_t plane_x = (size_t)p.n_tok * row_bytes;
    const uint32_t total = p.n_tok * (uint32_t)p.nvec;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const uint32_t g = fastdiv(i, p.div_nvec);
        const uint32_t v = i - g * (uint32_t)p.nvec;
        const uint32_t s = fastdiv(g, p.div_Tm);
        float a[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = 0.f;
        if ((int)(g - s * (uint32_t)p.Tm) < held(p, (int)s)) {
            const uint8_t *src = p.y + (size_t)g * row_bytes + (size_t)v * 16;
            for (int d0 = 0; d0 < p.W; d0 += 8) {
                uint4 x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (d0 + u < p.W) x[u] = ld_stream_v4(src + (size_t)(d0 + u) * plane_x);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (d0 + u >= p.W) break;
                    const uint32_t q[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float lo = __uint_as_float(q[j] << 16);
                        const float hi = __uint_as_float(q[j] & 0xFFFF0000u);
                        if (OUT_F32) {
                            a[2 * j] = __fadd_rn(a[2 * j], lo);
                            a[2 * j + 1] = __fadd_rn(a[2 * j + 1], hi);
                        } else {
                            a[2 * j] = bf16_round(__fadd_rn(a[2 * j], lo));
                            a[2 * j + 1] = bf16_round(__fadd_rn(a[2 * j + 1], hi));
                        }
                    }
                }
            }
        }
        // the output is written once and read by nothing here: streaming stores
        if (OUT_F32) {
            float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + (size_t)g * p.h +
                                                   (size_t)v * 8);
            __stcs(o, make_float4(a[0], a[1], a[2], a[3]));
            __stcs(o + 1, make_float4(a[4], a[5], a[6], a[7]));
        } else {
            uint4 o;
            o.x = pack_bf16x2(a[0], a[1]);
            o.y = pack_bf16x2(a[2], a[3]);
            o.z = pack_bf16x2(a[4], a[5]);
            o.w = pack_bf16x2(a[6], a[7]);
            __stcs(reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.out) + (size_t)g * row_bytes +
                                             (size_t)v * 16), o);
        }
    }
}

// One-wave grid sizes, per device: SMs x resident CTAs of each kernel.
struct Waves {
    int gather, experts, reduce_bf16, reduce_f32;
};
std::mutex g_mu;
bool g_have[kMaxDevices];
Waves g_waves[kMaxDevices];

cudaError_t waves_for(int dev, Waves *w) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_have[dev]) {
        int sms = 0, a = 0, b = 0, c = 0, f = 0;
        cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, agrs_gather_kernel, kThreads, 0);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, agrs_experts_kernel, kThreads, 0);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c, agrs_reduce_kernel<false>, kThreads, 0);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&f, agrs_reduce_kernel<true>, kThreads, 0);
        if (e != cudaSuccess) return e;
        g_waves[dev] = Waves{sms * (a > 0 ? a : 1), sms * (b > 0 ? b : 1), sms * (c > 0 ? c : 1),
                             sms * (f > 0 ? f : 1)};
        g_have[dev] = true;
    }
    *w = g_waves[dev];
    return cudaSuccess;
}

int grid_for(long long items, int per_block, int wave) {
    const long long need = (items + per_block - 1) / per_block;
    return (int)(need < wave ? (need > 0 ? need : 1) : wave);
}

bool aligned16(const void *ptr) { return reinterpret_cast<uintptr_t>(ptr) % 16 == 0; }

}  // namespace

extern "C" int ep_agrs(const ep_config_t *cfg, const int32_t *num_tokens, const void *a1,
                       const int32_t *topk_ids, const float *topk_weights,
                       const ep_agrs_buffers_t *buf, int32_t out_dtype, void *out, void *stream) {
    int32_t tok_cap = 0, S = 0, Ecap = 0;
    if (ep_capacities(cfg, &tok_cap, &S, &Ecap) != EP_OK) return EP_ERR_INVALID_ARG;
    if (cfg->x_dtype != EP_BF16 || (cfg->flags & EP_FLAG_WEIGHT_ON_INPUT)) return EP_ERR_INVALID_ARG;
    if (out_dtype != EP_BF16 && out_dtype != EP_F32) return EP_ERR_INVALID_ARG;
    if (!a1 || !topk_ids || !topk_weights || !buf || !buf->x_g || !buf->ids_g || !buf->w_g ||
        !buf->y || !out)
        return EP_ERR_INVALID_ARG;
    if (!aligned16(a1) || !aligned16(buf->x_g) || !aligned16(buf->y) || !aligned16(out))
        return EP_ERR_INVALID_ARG;
    const long long W = cfg->W, Tm = cfg->max_tokens, nvec = cfg->hidden / 8, K = cfg->top_k;
    // work items of each kernel stay within 2^31
    if (W * W * Tm * nvec >= (1LL << 31) || W * Tm * (nvec + K) >= (1LL << 31)) return EP_ERR_INVALID_ARG;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EP_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return EP_ERR_INVALID_ARG;
    Waves wv;
    if (waves_for(dev, &wv) != cudaSuccess) return EP_ERR_CUDA;

    AgrsParams p = {};
    p.a1 = static_cast<const uint8_t *>(a1);
    p.ids = topk_ids;
    p.weights = topk_weights;
    p.num_tokens = num_tokens;
    p.x_g = static_cast<uint8_t *>(buf->x_g);
    p.ids_g = buf->ids_g;
    p.w_g = buf->w_g;
    p.y = static_cast<uint8_t *>(buf->y);
    p.out = out;
    p.status = buf->status;
    p.W = cfg->W;
    p.E = cfg->E;
    p.K = cfg->top_k;
    p.Tm = cfg->max_tokens;
    p.e_local = cfg->E / cfg->W;
    p.h = cfg->hidden;
    p.nvec = (int)nvec;
    p.n_tok = (uint32_t)(W * Tm);
    p.div_nvec = make_fastdiv((uint32_t)nvec);
    p.div_K = make_fastdiv((uint32_t)K);
    p.div_Tm = make_fastdiv((uint32_t)Tm);
    p.div_ntok = make_fastdiv(p.n_tok);

    struct Range {   // NVTX range over the three launches
        Range() { nvtxRangePushA("ep:agrs"); }
        ~Range() { nvtxRangePop(); }
    } range;
    if (p.status && cudaMemsetAsync(p.status, 0, sizeof(int32_t), st) != cudaSuccess) return EP_ERR_CUDA;
    agrs_gather_kernel<<<grid_for(W * Tm * (nvec + K), kThreads, wv.gather), kThreads, 0, st>>>(p);
    if (cudaGetLastError() != cudaSuccess) return EP_ERR_CUDA;
    agrs_experts_kernel<<<grid_for(W * W * Tm, kWarps, wv.experts), kThreads, 0, st>>>(p);
    if (cudaGetLastError() != cudaSuccess) return EP_ERR_CUDA;
    if (out_dtype == EP_F32)
        agrs_reduce_kernel<true><<<grid_for(W * Tm * nvec, kThreads, wv.reduce_f32), kThreads, 0, st>>>(p);
    else
        agrs_reduce_kernel<false><<<grid_for(W * Tm * nvec, kThreads, wv.reduce_bf16), kThreads, 0, st>>>(p);
    if (cudaGetLastError() != cudaSuccess) return EP_ERR_CUDA;
    return EP_OK;
}
