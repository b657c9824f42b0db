// route.cu -- the routing kernel of the EP dispatch: one CTA per routing tile
// (see route_tile.cuh for what a tile computes and how), plus the per-launch
// bookkeeping: tiles take tickets in launch order, every tile reads the
// launch's look-back epoch from the device header, and the last CTA to finish
// rearms the ticket and advances the epoch for the next launch.
#include "route_tile.cuh"

namespace ep {

template <int KT>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(const RouteParams p) {
    extern __shared__ __align__(16) uint32_t sm[];
    __shared__ int s_tile;
    __shared__ uint32_t s_epoch;
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_tile = (int)atomicAdd(&p.hdr->ticket, 1u);
        // The epoch lives in device memory and only the launch's last CTA
        // advances it (after every CTA has read it), so every tile of one launch
        // reads the same value, and a replayed launch (a CUDA graph) gets a
        // fresh one without any host involvement. The previous launch's write is
        // ordered before this launch by the launch boundary: a relaxed load.
        s_epoch = ld_relaxed_u32(&p.hdr->epoch) & 0x3FFFFFFFu;
    }
    __syncthreads();
    // Every routing CTA is resident once it gets here, so a dependent kernel
    // launched early cannot starve a routing tile of an SM.
    pdl_launch_dependents();
    const int q = s_tile;
    const uint32_t epoch = s_epoch;
    if (q < p.num_tiles) {
        route_tile<KT>(p, q, epoch, sm);
    } else if (tid == 0) {
        raise_error(p.hdr, EP_ERR_STATE);   // a stale ticket counter; never expected
    }
    // the last CTA to finish rearms the ticket and advances the epoch
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(&p.hdr->done, 1u) == gridDim.x - 1) {
            atomicExch(&p.hdr->ticket, 0u);
            atomicExch(&p.hdr->done, 0u);
            atomicExch(&p.hdr->epoch, (epoch + 1u) & 0x3FFFFFFFu);
        }
    }
}

template <int KT>
static cudaError_t launch_route_kt(const RouteParams &p, size_t smem, cudaStream_t st) {
    cudaError_t e = ensure_dyn_smem((const void *)route_kernel<KT>, smem);
    if (e != cudaSuccess) return e;
    route_kernel<KT><<<p.num_tiles, kRouteThreads, smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_route(const RouteParams &p, cudaStream_t st) {
    const size_t smem = route_smem_bytes(p.n_ctr, p.K);
    switch (route_kt(p.K)) {
        case 1: return launch_route_kt<1>(p, smem, st);
        case 2: return launch_route_kt<2>(p, smem, st);
        case 4: return launch_route_kt<4>(p, smem, st);
        case 8: return launch_route_kt<8>(p, smem, st);
        case 16: return launch_route_kt<16>(p, smem, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ep
