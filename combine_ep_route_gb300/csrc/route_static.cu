// route_static.cu -- ep_route_static: the routing step of ep_dispatch with its
// scratch memory in a fixed, file-scope device array instead of a
// caller-provided workspace, for callers that cannot allocate device memory.
//
// The routing kernel needs scratch beyond its inputs and outputs: a status
// header (first error, tile ticket and completion counters), one look-back flag
// per routing tile, and two vectors of W+E counters per tile (its aggregate and
// its inclusive prefix). Here those live in g_route_scratch, a static
// __device__ array of EP_STATIC_SCRATCH_BYTES. Every GPU that loads this
// library holds that array until the process exits.
//
// In host code the name g_route_scratch is only a host-side stand-in for the
// device array: passing it to a kernel would make the kernel fault (or, where
// the GPU can reach host memory, silently use the wrong memory). The device
// address is therefore looked up once per device, with that device current,
// through cudaGetSymbolAddress, and that address is what the kernel gets.
#include "ep_internal.cuh"

#include <cstddef>
#include <cstdint>
#include <mutex>

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kRegionAlign = 256;

__device__ __align__(256) uint8_t g_route_scratch[EP_STATIC_SCRATCH_BYTES];

std::mutex g_mu;
uint8_t *g_scratch_dev[kMaxDevices];   // device address of g_route_scratch, per device

size_t align_region(size_t x) { return (x + kRegionAlign - 1) / kRegionAlign * kRegionAlign; }

// Copies the call's first device-side error (0 if none) to the caller's word.
__global__ void static_status_kernel(const ep::DevHeader *hdr, int32_t *status) {
    if (blockIdx.x == 0 && threadIdx.x == 0) *status = hdr->err;
}

}  // namespace

extern "C" int ep_route_static(const ep_config_t *cfg, const int32_t *num_tokens,
                               const int32_t *topk_ids, const float *topk_weights,
                               const ep_route_outputs_t *out, void *stream) {
    int32_t tok_cap = 0, S = 0, Ecap = 0;
    if (ep_capacities(cfg, &tok_cap, &S, &Ecap) != EP_OK) return EP_ERR_INVALID_ARG;
    if (!topk_ids || !topk_weights || !out || !out->send_cnt || !out->pair_row || !out->pair_w ||
        !out->pair_send || !out->recv_eloc || !out->recv_w || !out->recv_row ||
        !out->expert_num_tokens)
        return EP_ERR_INVALID_ARG;
    // every input and output is read or written as 4-byte words
    const void *words[] = {num_tokens,      topk_ids,       topk_weights,   out->send_cnt,
                           out->pair_row,   out->pair_w,    out->pair_send, out->recv_eloc,
                           out->recv_w,     out->recv_row,  out->expert_num_tokens, out->status};
    for (const void *p : words)
        if (reinterpret_cast<uintptr_t>(p) % 4 != 0) return EP_ERR_INVALID_ARG;

    // scratch this problem needs: header, tile flags, tile aggregates, tile prefixes
    const int W = cfg->W, Tm = cfg->max_tokens;
    const int tiles_per_rank = (Tm + ep::kRouteTile - 1) / ep::kRouteTile;
    const int num_tiles = W * tiles_per_rank;
    const int n_ctr = W + cfg->E;
    const size_t off_flag = align_region(sizeof(ep::DevHeader));
    const size_t off_agg = off_flag + align_region((size_t)num_tiles * ep::kFlagStride * 4);
    const size_t off_incl = off_agg + align_region((size_t)num_tiles * n_ctr * 4);
    const size_t need = off_incl + align_region((size_t)num_tiles * n_ctr * 4);
    if (need > (size_t)EP_STATIC_SCRATCH_BYTES) return EP_ERR_SCRATCH_LIMIT;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the caller's status word says "no error" until the routing kernel has run
    if (out->status && cudaMemsetAsync(out->status, 0, sizeof(int32_t), st) != cudaSuccess)
        return EP_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EP_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return EP_ERR_INVALID_ARG;

    uint8_t *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_scratch_dev[dev]) {
            // set-up, once per device, with that device current
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return EP_ERR_CUDA;
            g_scratch_dev[dev] = static_cast<uint8_t *>(p);
        }
        scratch = g_scratch_dev[dev];
    }
    // The header's first error, tile ticket and completion count must start at
    // zero; the array keeps whatever the previous call left in it. Its look-back
    // epoch is kept: the kernel advances it, so flags left by earlier calls
    // (which carry older epochs) never look current.
    if (cudaMemsetAsync(scratch, 0, offsetof(ep::DevHeader, epoch), st) != cudaSuccess)
        return EP_ERR_CUDA;

    ep::RouteParams rp = {};
    rp.ids = topk_ids;
    rp.weights = topk_weights;
    rp.num_tokens = num_tokens;
    rp.W = W;
    rp.E = cfg->E;
    rp.K = cfg->top_k;
    rp.Tm = Tm;
    rp.e_local = cfg->E / W;
    rp.S = S;
    rp.Ecap = Ecap;
    rp.tiles_per_rank = tiles_per_rank;
    rp.num_tiles = num_tiles;
    rp.n_ctr = n_ctr;
    rp.hdr = reinterpret_cast<ep::DevHeader *>(scratch);
    rp.tile_flag = reinterpret_cast<uint32_t *>(scratch + off_flag);
    rp.tile_agg = reinterpret_cast<int32_t *>(scratch + off_agg);
    rp.tile_incl = reinterpret_cast<int32_t *>(scratch + off_incl);
    rp.send_cnt = out->send_cnt;
    rp.pair_row = out->pair_row;
    rp.pair_w = out->pair_w;
    rp.pair_send = out->pair_send;
    rp.recv_eloc = out->recv_eloc;
    rp.recv_w = out->recv_w;
    rp.recv_row = out->recv_row;
    rp.expert_num_tokens = out->expert_num_tokens;
    rp.wait_limit_ns = 2000000000ull;
    rp.fault_skip_tile = -1;
    rp.vec_ids = (reinterpret_cast<uintptr_t>(topk_ids) % 16 == 0) &&
                 (reinterpret_cast<uintptr_t>(topk_weights) % 16 == 0);
    rp.unit_weights = (cfg->flags & EP_FLAG_WEIGHT_ON_INPUT) ? 1 : 0;
    rp.vec_recv = S % 4 == 0 && reinterpret_cast<uintptr_t>(out->recv_eloc) % 16 == 0 &&
                  reinterpret_cast<uintptr_t>(out->recv_w) % 16 == 0 &&
                  reinterpret_cast<uintptr_t>(out->recv_row) % 16 == 0;
    if (ep::launch_route(rp, st) != cudaSuccess) return EP_ERR_CUDA;
    if (out->status) {
        static_status_kernel<<<1, 32, 0, st>>>(rp.hdr, out->status);
        if (cudaGetLastError() != cudaSuccess) return EP_ERR_CUDA;
    }
    return EP_OK;
}
