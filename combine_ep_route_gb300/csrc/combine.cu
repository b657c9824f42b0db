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
// One thread produces 16 bytes of bf16 input (8 elements) of one token: it
// reads its token's row indices and weights (shared by the threads of the
// token through L1), issues all top_k 16-byte loads before using any, then
// folds. Expert rows are streamed (no L1 allocation); HBM sees each pair row
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

template <int KMAX, bool OUT_F32>
__global__ void __launch_bounds__(256) combine_kernel(const CombineParams p) {
    pdl_wait();   // expert_out may be the previous kernel's output
    const int nvec = p.nvec, K = p.K;
    const uint32_t total = (uint32_t)p.n_tokens * (uint32_t)nvec;   // < 2^31
    const size_t row_bytes = (size_t)p.h * 2;
    for (uint32_t idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += gridDim.x * blockDim.x) {
        const int g = (int)fastdiv(idx, p.div_nvec);
        const int v = (int)(idx - (uint32_t)g * (uint32_t)nvec);
        int32_t r[KMAX];
        float w[KMAX];
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            r[k] = k < K ? __ldg(p.pair_row + (size_t)g * K + k) : -1;
            if (r[k] >= p.n_rows) r[k] = -1;   // routing never writes such a row
            w[k] = k < K ? __ldg(p.pair_w + (size_t)g * K + k) : 0.f;
        }
        uint4 x[KMAX];
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            if (r[k] >= 0) x[k] = ld_stream_v4(p.expert_out + (size_t)r[k] * row_bytes + (size_t)v * 16);
            else x[k] = make_uint4(0u, 0u, 0u, 0u);
        }
        float a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = 0.f;
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            if (r[k] < 0) continue;
            fold2(a[0], a[1], w[k], x[k].x);
            fold2(a[2], a[3], w[k], x[k].y);
            fold2(a[4], a[5], w[k], x[k].z);
            fold2(a[6], a[7], w[k], x[k].w);
        }
        if (OUT_F32) {
            float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + (size_t)g * p.h +
                                                   (size_t)v * 8);
            o[0] = make_float4(a[0], a[1], a[2], a[3]);
            o[1] = make_float4(a[4], a[5], a[6], a[7]);
        } else {
            uint4 o;
            o.x = pack_bf16x2(a[0], a[1]);
            o.y = pack_bf16x2(a[2], a[3]);
            o.z = pack_bf16x2(a[4], a[5]);
            o.w = pack_bf16x2(a[6], a[7]);
            *reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.out) + (size_t)g * row_bytes +
                                       (size_t)v * 16) = o;
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
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv;
             i += (size_t)gridDim.x * blockDim.x)
            base[i] = make_uint4(0u, 0u, 0u, 0u);
    }
}

cudaError_t launch_zero_pad(const ZeroPadParams &p, int grid_x, cudaStream_t st) {
    zero_pad_kernel<<<dim3(grid_x, p.E), 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ep
