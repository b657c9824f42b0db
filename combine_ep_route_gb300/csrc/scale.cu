// scale.cu -- dispatch with apply_router_weight_on_input.
//
// `prepare` of vLLM AllToAllBatchedPrepareAndFinalize allows, for top_k == 1,
// that the router weight is applied on the way in: a1 = a1 * topk_weights
// converted to the activation type, and the weights carried on become one. Each
// token then has at most one destination row, and the row must be scaled while
// it moves, which the bulk-copy mover cannot do. This kernel does it in
// registers: one thread per 16 bytes of a token's row, every element rounded
// as the page's bf16 product rounds it, bf16(x * bf16(w)) (the product of two
// bf16 values is exact in fp32, so one rounding). Extra payload bytes travel
// unscaled. The destination is the token's b_a1 row (fused path) or its send
// row (send-buffer path, then exchanged and delivered by the mover).
#include "ep_internal.cuh"

#include <cuda_bf16.h>

namespace ep {

namespace {

__device__ __forceinline__ uint32_t scale2(uint32_t x, float w) {
    const float lo = __fmul_rn(__uint_as_float(x << 16), w);
    const float hi = __fmul_rn(__uint_as_float(x & 0xFFFF0000u), w);
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

}  // namespace

__global__ void __launch_bounds__(256) scale_move_kernel(const ScaleMoveParams p) {
    for (uint32_t idx = blockIdx.x * blockDim.x + threadIdx.x; idx < p.n_items;
         idx += gridDim.x * blockDim.x) {
        const uint32_t g = fastdiv(idx, p.div_vecs);   // token
        const uint32_t v = idx - g * p.vecs;          // 16-byte vector of its row (+ extras)
        const int drow = __ldg(p.dst_index + g);     // top_k == 1: one pair per token
        if (drow < 0 || drow >= p.n_dst_rows) continue;
        if (v < p.nvec_a1) {
            const uint4 x = __ldg(reinterpret_cast<const uint4 *>(p.a1 + (size_t)g * p.a1_bytes) + v);
            const float w = __bfloat162float(__float2bfloat16_rn(__ldg(p.weights + g)));
            uint4 y;
            y.x = scale2(x.x, w);
            y.y = scale2(x.y, w);
            y.z = scale2(x.z, w);
            y.w = scale2(x.w, w);
            reinterpret_cast<uint4 *>(p.dst[0] + (size_t)drow * p.dst_stride[0])[v] = y;
        } else {
            // extra payload vectors: plain copies into their own rows (split) or
            // behind the activation in the same row (combined)
            uint32_t r = v - p.nvec_a1;
            int sg = 1;
            while (sg < p.n_seg && r >= p.seg_vecs[sg]) {
                r -= p.seg_vecs[sg];
                ++sg;
            }
            const uint4 x = __ldg(reinterpret_cast<const uint4 *>(p.src_seg[sg] +
                                                                 (size_t)g * p.seg_vecs[sg] * 16) + r);
            uint8_t *row = p.combined ? p.dst[0] + (size_t)drow * p.dst_stride[0] + p.seg_off[sg]
                                      : p.dst[sg] + (size_t)drow * p.dst_stride[sg];
            reinterpret_cast<uint4 *>(row)[r] = x;
        }
    }
}

cudaError_t launch_scale_move(const ScaleMoveParams &p, int grid, cudaStream_t st) {
    scale_move_kernel<<<grid, 256, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ep
