// combine.cu -- the weighted combine of the EP path, and the optional zero fill
// of unused batched-expert rows.
//
// Combine restates `finalize` of vLLM AllToAllBatchedPrepareAndFinalize for all
// W simulated ranks in one pass: every output row gathers the (at most top_k)
// expert-output rows its token was delivered to and sums them, weighted by the
// router weights. Because all ranks share one memory, the page's three steps
// (per-rank weighted partials, the return all_to_all_single, the per-token sum)
// collapse into one gather-reduce with no intermediate buffer. The fold is
// fp32 in top-k order, one rounded product and one rounded sum per pair
// (__fmul_rn / __fadd_rn, never contracted into an FMA), rounded once to the
// output type.
//
// One thread produces 16 bytes of bf16 input (8 elements) of one token -- or
// 2 or 4 such vectors when top_k is at most 4 or 2: it reads its token's row
// indices and weights (shared by the threads of the token through L1; 16-byte
// loads when top_k is a multiple of 4, which trimmed the prefill and Zipf
// combines by ~0.9 us on GB300), issues
// all its 16-byte loads before using any, then folds. Expert rows are streamed (no L1 allocation); HBM sees each pair row
// read once and each output row written once.
#include "ep_internal.cuh"

#include <cuda_bf16.h>

namespace ep {

namespace {

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void fold2(float &a0, float &a1, float w, uint32_t x) {
    const float lo = __uint_as_float(x << 16);
    const float hi = __uint_as_float(x & 0xFFFF0000u);
    a0 = __fadd_rn(a0, __fmul_rn(w, lo));
    a1 = __fadd_rn(a1, __fmul_rn(w, hi));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

}  // namespace

// Vectors per thread: a thread keeps about eight 16-byte loads in flight
// whatever top_k is (top_k 1: a thread reading one vector left HBM idle).
__host__ __device__ constexpr int vectors_per_thread(int kmax) { return kmax <= 2 ? 4 : (kmax <= 4 ? 2 : 1); }

template <int KMAX, bool OUT_F32>
__global__ void __launch_bounds__(256) combine_kernel(const CombineParams p) {
    constexpr int V = vectors_per_thread(KMAX);
    pdl_wait();   // expert_out may be the previous kernel's output
    const int nvec = p.nvec, K = p.K, G = p.groups;
    const uint32_t total = (uint32_t)p.n_tokens * (uint32_t)G;   // < 2^31
    const size_t row_bytes = (size_t)p.h * 2;
    for (uint32_t idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += gridDim.x * blockDim.x) {
        const int g = (int)fastdiv(idx, p.div_groups);
        const int q = (int)(idx - (uint32_t)g * (uint32_t)G);   // vectors q, q + G, ...
        int32_t r[KMAX];
        float w[KMAX];
        if (KMAX % 4 == 0 && K == KMAX) {   // 16-byte loads of the item's rows and weights
            const int4 *pr = reinterpret_cast<const int4 *>(p.pair_row + (size_t)g * KMAX);
            const float4 *pw = reinterpret_cast<const float4 *>(p.pair_w + (size_t)g * KMAX);
#pragma unroll
            for (int v = 0; v < KMAX / 4; ++v) {
                const int4 a = __ldg(pr + v);
                const float4 b = __ldg(pw + v);
                r[4 * v] = a.x, r[4 * v + 1] = a.y, r[4 * v + 2] = a.z, r[4 * v + 3] = a.w;
                w[4 * v] = b.x, w[4 * v + 1] = b.y, w[4 * v + 2] = b.z, w[4 * v + 3] = b.w;
            }
#pragma unroll
            for (int k = 0; k < KMAX; ++k)
                if (r[k] >= p.n_rows) r[k] = -1;
        } else {
#pragma unroll
            for (int k = 0; k < KMAX; ++k) {
                r[k] = k < K ? __ldg(p.pair_row + (size_t)g * K + k) : -1;
                if (r[k] >= p.n_rows) r[k] = -1;   // routing never writes such a row
                w[k] = k < K ? __ldg(p.pair_w + (size_t)g * K + k) : 0.f;
            }
        }
        uint4 x[KMAX][V];
#pragma unroll
        for (int k = 0; k < KMAX; ++k)
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int v = q + j * G;
                if (r[k] >= 0 && v < nvec)
                    x[k][j] = ld_stream_v4(p.expert_out + (size_t)r[k] * row_bytes + (size_t)v * 16);
                else
                    x[k][j] = make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int v = q + j * G;
            if (v >= nvec) break;
            float a[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = 0.f;
#pragma unroll
            for (int k = 0; k < KMAX; ++k) {
                if (r[k] < 0) continue;
                fold2(a[0], a[1], w[k], x[k][j].x);
                fold2(a[2], a[3], w[k], x[k][j].y);
                fold2(a[4], a[5], w[k], x[k][j].z);
                fold2(a[6], a[7], w[k], x[k][j].w);
            }
            // the output is written once and read by nothing here: streaming
            // (evict-first) stores (measured on GB300: prefill combine 163.6 ->
            // 162.0 us, Zipf 96.3 -> 93.2, grouped 145.2 -> 142.9, decode unchanged;
            // an evict-first policy on the row loads instead changed nothing)
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
}

template <int KMAX>
static const void *pick_combine(bool out_f32) {
    return out_f32 ? (const void *)combine_kernel<KMAX, true> : (const void *)combine_kernel<KMAX, false>;
}

static const void *combine_fn(int K, bool out_f32) {
    if (K <= 2) return pick_combine<2>(out_f32);
    if (K <= 4) return pick_combine<4>(out_f32);
    if (K <= 8) return pick_combine<8>(out_f32);
    return pick_combine<16>(out_f32);
}

int combine_vectors_per_thread(int top_k) {
    return vectors_per_thread(top_k <= 2 ? 2 : (top_k <= 4 ? 4 : (top_k <= 8 ? 8 : 16)));
}

// Resident CTAs per SM of the combine kernel for this top_k (one full wave of
// the persistent grid).
cudaError_t combine_occupancy(int top_k, bool out_f32, int *ctas_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, combine_fn(top_k, out_f32), 256, 0);
}

cudaError_t launch_combine(const CombineParams &p, bool out_f32, int grid, bool pdl,
                           cudaStream_t st) {
    const void *fn = combine_fn(p.K, out_f32);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<CombineParams *>(&p)};
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Two-stage combine: `finalize` of AllToAllBatchedPrepareAndFinalize in the
// page's own rounding. Stage 1 runs on the receiving side of every rank: for
// each received slot it weights the slot's columns (their expert-output rows)
// and sums them in fp32, columns in order, then rounds the partial to bf16 --
// the payload the page sends back with all_to_all_single. Stage 2 runs on the
// sending side: each token sums the partials of the ranks it went to, ranks in
// ascending order, in the output type (bf16: every sum rounded; fp32: fp32
// sums). The exchange between the stages is no copy here: stage 2 reads the
// other rank's block of the stage-1 buffer directly.
template <int ST>   // slots per token rounded up to a power of two
__global__ void __launch_bounds__(256) combine_partial_kernel(const PartialParams p) {
    // one warp per received slot row (d, s, slot); lanes share its column list
    const int lane = threadIdx.x & 31;
    const uint32_t n_rows = (uint32_t)p.W * p.W * p.Tm;
    const size_t row_bytes = (size_t)p.h * 2;
    for (uint32_t r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < n_rows;
         r += (gridDim.x * blockDim.x) >> 5) {
        const uint32_t ds = fastdiv(r, p.div_tm);              // d * W + s
        const int slot = (int)(r - ds * (uint32_t)p.Tm);
        const int d = (int)fastdiv(ds, p.div_w);
        const int s = (int)(ds - (uint32_t)d * (uint32_t)p.W);
        if (slot >= __ldg(p.send_cnt + s * p.W + d)) continue;   // warp-uniform
        const size_t base = (size_t)r * p.S;
        int64_t my_src = -1;
        float my_w = 0.f;
        if (lane < p.S) {
            const int j = __ldg(p.recv_eloc + base + lane);
            const int row = __ldg(p.recv_row + base + lane);
            if (j >= 0 && j < p.e_local && row >= 0 && row < p.Ecap) {
                my_src = (int64_t)(d * p.e_local + j) * p.Ecap + row;
                my_w = __ldg(p.recv_w + base + lane);
            }
        }
        // the valid columns, compacted in column order (the fold order); a
        // column's row and weight stay in the lane that read them and are
        // fetched by shuffle where they are used, which keeps registers free
        // for more warps in flight
        const uint32_t vmask = __ballot_sync(0xffffffffu, my_src >= 0);
        const int nv = __popc(vmask);
        uint8_t *dst = p.part + (size_t)r * p.part_stride;
        // four vectors per lane per round; two columns' loads go out together, so
        // a slot with several columns keeps twice the bytes in flight. The rounds
        // are counted per warp, not per lane, so that every lane takes part in
        // every shuffle below even when a row is shorter than the warp's span.
        for (int vb = 0; vb < p.nvec; vb += 128) {
            const int v0 = vb + lane;
            float a[4][8];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int i = 0; i < 8; ++i) a[u][i] = 0.f;
#pragma unroll
            for (int c = 0; c < ST; c += 2) {
                if (c >= nv) break;
                const bool two = c + 1 < nv;
                const int from0 = __fns(vmask, 0, c + 1);
                const int from1 = two ? __fns(vmask, 0, c + 2) : from0;
                const int64_t src0 = __shfl_sync(0xffffffffu, my_src, from0);
                const int64_t src1 = __shfl_sync(0xffffffffu, my_src, from1);
                const float w0 = __shfl_sync(0xffffffffu, my_w, from0);
                const float w1 = __shfl_sync(0xffffffffu, my_w, from1);
                const uint8_t *row0 = p.expert_out + (size_t)src0 * row_bytes;
                const uint8_t *row1 = p.expert_out + (size_t)src1 * row_bytes;
                uint4 x[2][4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int v = v0 + 32 * u;
                    const bool in = v < p.nvec;
                    x[0][u] = in ? ld_stream_v4(row0 + (size_t)v * 16) : make_uint4(0u, 0u, 0u, 0u);
                    x[1][u] = in && two ? ld_stream_v4(row1 + (size_t)v * 16) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    if (q == 1 && !two) break;
                    const float wc = q == 0 ? w0 : w1;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        fold2(a[u][0], a[u][1], wc, x[q][u].x);
                        fold2(a[u][2], a[u][3], wc, x[q][u].y);
                        fold2(a[u][4], a[u][5], wc, x[q][u].z);
                        fold2(a[u][6], a[u][7], wc, x[q][u].w);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int v = v0 + 32 * u;
                if (v >= p.nvec) break;
                uint4 o;
                o.x = pack_bf16x2(a[u][0], a[u][1]);
                o.y = pack_bf16x2(a[u][2], a[u][3]);
                o.z = pack_bf16x2(a[u][4], a[u][5]);
                o.w = pack_bf16x2(a[u][6], a[u][7]);
                *reinterpret_cast<uint4 *>(dst + (size_t)v * 16) = o;
            }
        }
    }
}

__device__ __forceinline__ float round_bf16(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}

// acc += two bf16 partials: an fp32 sum, or a bf16 sum rounded after each add.
template <bool OUT_F32>
__device__ __forceinline__ void add2(float &a0, float &a1, uint32_t x) {
    const float lo = __uint_as_float(x << 16);
    const float hi = __uint_as_float(x & 0xFFFF0000u);
    if (OUT_F32) {
        a0 = __fadd_rn(a0, lo);
        a1 = __fadd_rn(a1, hi);
    } else {
        a0 = round_bf16(__fadd_rn(a0, lo));
        a1 = round_bf16(__fadd_rn(a1, hi));
    }
}

// Two bf16 sums at once, each rounded to nearest even. For bf16 operands this
// gives the same bits as an fp32 sum rounded to bf16: the fp32 sum is exact
// whenever the exponents differ by at most 15, and otherwise the smaller
// operand lies far below half a bf16 unit of the larger, so both roundings
// return the larger.
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ void cmp_swap(int &a, int &b) {
    const int lo = min(a, b), hi = max(a, b);
    a = lo;
    b = hi;
}

// Ascending sort of N register values: an optimal 19-exchange network for 8
// (Knuth, TAOCP vol. 3, 5.3.4), insertion sort otherwise.
template <int N>
__device__ __forceinline__ void sort_ascending(int (&v)[N]) {
    if constexpr (N == 8) {
        cmp_swap(v[0], v[2]); cmp_swap(v[1], v[3]); cmp_swap(v[4], v[6]); cmp_swap(v[5], v[7]);
        cmp_swap(v[0], v[4]); cmp_swap(v[1], v[5]); cmp_swap(v[2], v[6]); cmp_swap(v[3], v[7]);
        cmp_swap(v[0], v[1]); cmp_swap(v[2], v[3]); cmp_swap(v[4], v[5]); cmp_swap(v[6], v[7]);
        cmp_swap(v[2], v[4]); cmp_swap(v[3], v[5]);
        cmp_swap(v[1], v[4]); cmp_swap(v[3], v[6]);
        cmp_swap(v[1], v[2]); cmp_swap(v[3], v[4]); cmp_swap(v[5], v[6]);
    } else {
#pragma unroll
        for (int i = 1; i < N; ++i)
#pragma unroll
            for (int k = i; k > 0; --k) cmp_swap(v[k - 1], v[k]);
    }
}

template <int KT, bool OUT_F32>
__global__ void __launch_bounds__(256) combine_gather_kernel(const GatherParams p) {
    // one thread per 16 bytes of bf16 input of one token: the token's send rows
    // (at most one per destination rank) sorted ascending -- ascending rank --
    // then every partial's load issued before the sum
    for (uint32_t idx = blockIdx.x * blockDim.x + threadIdx.x; idx < p.n_items;
         idx += gridDim.x * blockDim.x) {
        const uint32_t g = fastdiv(idx, p.div_nvec);
        const uint32_t v = idx - g * (uint32_t)p.nvec;
        const int s = (int)fastdiv(g, p.div_tm);
        int sr[KT];
#pragma unroll
        for (int k = 0; k < KT; ++k) {
            const int x = k < p.K ? __ldg(p.pair_send + (size_t)g * p.K + k) : -1;
            sr[k] = x < 0 ? 0x7FFFFFFF : x;
        }
        sort_ascending<KT>(sr);
        uint4 x[KT];
        bool has[KT];
#pragma unroll
        for (int k = 0; k < KT; ++k) {   // the partial row of each destination, in the rank-d block
            has[k] = false;
            x[k] = make_uint4(0u, 0u, 0u, 0u);
            if (sr[k] != 0x7FFFFFFF) {
                const uint32_t sd = fastdiv((uint32_t)sr[k], p.div_tm);   // s * W + d
                const int slot = (int)((uint32_t)sr[k] - sd * (uint32_t)p.Tm);
                const int d = (int)(sd - (uint32_t)s * (uint32_t)p.W);
                if (d >= 0 && d < p.W) {
                    const size_t rrow = ((size_t)d * p.W + s) * p.Tm + slot;
                    x[k] = ld_stream_v4(p.part + rrow * p.part_stride + (size_t)v * 16);
                    has[k] = true;
                }
            }
        }
        if (OUT_F32) {
            float a[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = 0.f;
#pragma unroll
            for (int k = 0; k < KT; ++k) {   // destinations in ascending rank order
                if (!has[k]) continue;
                add2<true>(a[0], a[1], x[k].x);
                add2<true>(a[2], a[3], x[k].y);
                add2<true>(a[4], a[5], x[k].z);
                add2<true>(a[6], a[7], x[k].w);
            }
            float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + (size_t)g * p.h +
                                                   (size_t)v * 8);
            __stcs(o, make_float4(a[0], a[1], a[2], a[3]));   // streaming, as in combine_kernel
            __stcs(o + 1, make_float4(a[4], a[5], a[6], a[7]));
        } else {
            // bf16 sums, each rounded, in ascending rank order: native bf16 adds
            // (see add_bf16x2), starting from +0 like the fp32 form
            uint4 o = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int k = 0; k < KT; ++k) {
                if (!has[k]) continue;
                o.x = add_bf16x2(o.x, x[k].x);
                o.y = add_bf16x2(o.y, x[k].y);
                o.z = add_bf16x2(o.z, x[k].z);
                o.w = add_bf16x2(o.w, x[k].w);
            }
            __stcs(reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.out) + (size_t)g * p.h * 2 +
                                             (size_t)v * 16), o);
        }
    }
}

// One-wave grid (SMs x resident CTAs) for a kernel, capped by its work.
static int wave_grid(const void *fn, int num_sms, uint32_t items) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, 256, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    const long long need = ((long long)items + 255) / 256;
    const long long wave = (long long)num_sms * per_sm;
    return (int)(need < 1 ? 1 : (need < wave ? need : wave));
}

template <int ST>
static cudaError_t launch_partial_st(const PartialParams &a, int num_sms, cudaStream_t st) {
    const void *fn = (const void *)combine_partial_kernel<ST>;
    combine_partial_kernel<ST><<<wave_grid(fn, num_sms, a.n_items), 256, 0, st>>>(a);
    return cudaGetLastError();
}

template <int KT>
static cudaError_t launch_gather_kt(const GatherParams &b, bool out_f32, int num_sms, cudaStream_t st) {
    if (out_f32) {
        const void *fn = (const void *)combine_gather_kernel<KT, true>;
        combine_gather_kernel<KT, true><<<wave_grid(fn, num_sms, b.n_items), 256, 0, st>>>(b);
    } else {
        const void *fn = (const void *)combine_gather_kernel<KT, false>;
        combine_gather_kernel<KT, false><<<wave_grid(fn, num_sms, b.n_items), 256, 0, st>>>(b);
    }
    return cudaGetLastError();
}

cudaError_t launch_combine_two_stage(const PartialParams &a, const GatherParams &b, bool out_f32,
                                     int num_sms, cudaStream_t st) {
    cudaError_t e;
    if (a.S <= 2) e = launch_partial_st<2>(a, num_sms, st);
    else if (a.S <= 4) e = launch_partial_st<4>(a, num_sms, st);
    else if (a.S <= 8) e = launch_partial_st<8>(a, num_sms, st);
    else e = launch_partial_st<16>(a, num_sms, st);
    if (e != cudaSuccess) return e;
    if (b.K <= 2) return launch_gather_kt<2>(b, out_f32, num_sms, st);
    if (b.K <= 4) return launch_gather_kt<4>(b, out_f32, num_sms, st);
    if (b.K <= 8) return launch_gather_kt<8>(b, out_f32, num_sms, st);
    return launch_gather_kt<16>(b, out_f32, num_sms, st);
}

// Zero the rows of every expert at or past its row count, in every segment
// (b_a1 and the extra outputs), as the page's zero-filled batched buffer.
__global__ void __launch_bounds__(256) zero_pad_kernel(const ZeroPadParams p) {
    const int e = blockIdx.y;
    int n = p.expert_num_tokens[e];
    if (n < 0) n = 0;
    if (n > p.Ecap) n = p.Ecap;
    for (int sg = 0; sg < p.n_seg; ++sg) {
        const size_t bytes = p.seg_bytes[sg];
        uint4 *base = reinterpret_cast<uint4 *>(p.dst_seg[sg] + ((size_t)e * p.Ecap + n) * bytes);
        const size_t nv = (size_t)(p.Ecap - n) * bytes / 16;
        // streaming stores: the zeros are not read back by this step (measured on
        // GB300: zero-filled prefill step 4371 -> 4317 us)
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv;
             i += (size_t)gridDim.x * blockDim.x)
            __stcs(base + i, make_uint4(0u, 0u, 0u, 0u));
    }
}

// Received slots at or past a source's count get the page's fill: local id -1,
// weight 0, row -1 (its send_eloc / send_w start as full(-1) / zeros).
__global__ void __launch_bounds__(256) sanitize_recv_kernel(const ZeroPadParams p) {
    const size_t n = (size_t)p.W * p.W * p.Tm;
    for (size_t r = (size_t)blockIdx.x * blockDim.x + threadIdx.x; r < n;
         r += (size_t)gridDim.x * blockDim.x) {
        const int slot = (int)(r % p.Tm);
        const size_t ds = r / p.Tm;
        const int d = (int)(ds / p.W), s = (int)(ds % p.W);
        if (slot < p.send_cnt[s * p.W + d]) continue;
        for (int c = 0; c < p.S; ++c) {
            p.recv_eloc[r * p.S + c] = -1;
            p.recv_w[r * p.S + c] = 0.f;
            p.recv_row[r * p.S + c] = -1;
        }
    }
}

cudaError_t launch_zero_pad(const ZeroPadParams &p, int grid_x, cudaStream_t st) {
    zero_pad_kernel<<<dim3(grid_x, p.E), 256, 0, st>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    sanitize_recv_kernel<<<grid_x * 8, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ep
