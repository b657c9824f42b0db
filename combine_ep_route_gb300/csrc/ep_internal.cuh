// ep_internal.cuh -- shared definitions of the EP dispatch/combine library:
// workspace layout, kernel parameter blocks, device error reporting and the
// inline-PTX wrappers (mbarrier, bulk async copies, acquire/release flags,
// programmatic dependent launch) the sm_103a kernels use.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/ep.h"
#include "smem_limit.h"

namespace ep {

// ----------------------------------------------------------------- constants
constexpr int kRouteTile = 64;                  // tokens per routing tile
constexpr int kRouteThreads = 256;              // threads per routing CTA (4 per token)
constexpr int kRouteWarps = kRouteTile / 32;    // warps that hold one token each per lane
constexpr int kAlign = 256;                     // workspace sub-buffer alignment
constexpr int kMaxDst = EP_MAX_TOPK;            // destinations of one row, at most
constexpr int kMaxSeg = 1 + EP_MAX_EXTRA;       // a1 + extra payloads
constexpr uint32_t kMoveSmemBudget = 200 * 1024;  // stage memory of one mover CTA
// Each routing tile's flag sits on its own 128-byte line: the flags are polled
// by the look-back of later tiles and by the row movers, and on one shared
// line those polls would queue the tiles' own release stores behind them.
constexpr int kFlagStride = 32;                 // uint32 words between two tiles' flags

// Device-side status block at the start of the workspace.
struct DevHeader {
    int32_t err;          // first EP_ERR_* raised on the device, 0 if none
    uint32_t err_count;   // how many raises since the last ep_status
    uint32_t ticket;      // routing tiles started in this launch (reset by the last tile)
    uint32_t done;        // routing tiles finished in this launch
    uint32_t epoch;       // look-back epoch of the running launch; the last tile advances it
    uint32_t move_next;   // next row-mover unit handed out (fused dispatch; reset at the end)
    uint32_t routers;     // CTAs of the fused dispatch that asked to route (reset at the end)
    uint32_t pad[57];
};
static_assert(sizeof(DevHeader) == 256, "header is one aligned block");

// Byte offsets of the workspace sub-buffers.
struct Layout {
    size_t hdr, tile_flag, tile_agg, tile_incl, send_cnt, pair_row, pair_w, pair_send,
        recv_eloc, recv_w, recv_row, send_x, recv_x, total;
    int num_tiles, tiles_per_rank, n_ctr, S, Ecap, e_local;
    uint32_t row_bytes;   // a1 row + extra rows, one send-buffer row
};

// ------------------------------------------------------------ parameter blocks
struct RouteParams {
    const int32_t *ids;
    const float *weights;
    const int32_t *num_tokens;   // may be null
    int W, E, K, Tm, e_local, S, Ecap, tiles_per_rank, num_tiles, n_ctr;
    DevHeader *hdr;
    uint32_t *tile_flag;
    int32_t *tile_agg, *tile_incl;
    int32_t *send_cnt, *pair_row, *pair_send, *recv_eloc, *recv_row;
    float *pair_w, *recv_w;
    int32_t *expert_num_tokens;
    uint64_t wait_limit_ns;
    int32_t fault_skip_tile;
    int32_t route_ctas;          // fused dispatch: CTAs that route (the first to arrive); 0 = all
    int32_t vec_ids;             // ids and weights 16-byte aligned: vector loads allowed
    int32_t vec_recv;            // S % 4 == 0 and recv_* 16-byte aligned: vector row stores
    int32_t unit_weights;        // weights applied on input: carry 1.0 instead of w
};

// Division by a run-time invariant d via multiply and shift (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994):
// for d >= 1 and 0 <= n < 2^31, n / d == (umulhi(n, m) + n) >> l with
// l = ceil(log2 d) and m = floor(2^32 * (2^l - d) / d) + 1.
struct FastDiv {
    uint32_t d, m, l;
};

inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    f.d = d;
    f.l = 0;
    while ((1ull << f.l) < d) ++f.l;
    f.m = (uint32_t)((((1ull << f.l) - d) << 32) / d + 1);
    return f;
}

__device__ __forceinline__ uint32_t fastdiv(uint32_t n, const FastDiv &f) {
    return (__umulhi(n, f.m) + n) >> f.l;
}

enum MoveMode { MOVE_FUSED = 0, MOVE_PACK = 1, MOVE_EXCHANGE = 2, MOVE_DELIVER = 3 };

struct MoveParams {
    int W, K, Tm, S, e_local, Ecap;
    int n_seg;                          // 1 + n_extra
    uint32_t seg_bytes[kMaxSeg];        // bytes of each payload segment
    uint32_t seg_off[kMaxSeg];          // offset of each segment in a combined row
    uint32_t row_bytes;                 // combined row (sum of segments)
    int chunks;                         // a1 part of a row moved as this many units
    uint32_t chunk_bytes;               // seg_bytes[0] / chunks (multiple of 16)
    const uint8_t *src_seg[kMaxSeg];    // token-major sources [W*Tm][seg_bytes]
    uint8_t *dst_seg[kMaxSeg];          // expert-major outputs [E*Ecap][seg_bytes]
    uint8_t *send_x, *recv_x;           // [W*W*Tm][row_bytes]
    const int32_t *pair_row, *pair_send, *send_cnt, *recv_eloc, *recv_row;
    int n_tokens;                       // W*Tm
    int n_rows;                         // E*Ecap rows of the batched layout
    int n_slots;                        // W*W*Tm send-buffer rows
    int pipes;                          // warps of a CTA that run a pipeline (the rest idle)
    int stages;                         // stages per pipeline
    uint32_t stage_bytes;
    DevHeader *hdr;
    uint64_t wait_limit_ns;
    // routing in the same launch: wait for a token's tile before reading its rows
    int wait_tiles;
    int dynamic_units;                  // warps grab units from hdr->move_next
    const uint32_t *tile_flag;
    int tiles_per_rank;
    FastDiv div_tm;
};

// One-launch dispatch of a small batch (dispatch_small.cu): every CTA owns
// n_per consecutive token slots and counts its own prefix.
constexpr int kSmallMaxTokens = 32;    // token slots per CTA, at most (one lane bit each)
constexpr int kSmallMaxIds = 16384;    // W * max_tokens * top_k, at most (ids every CTA may read)

struct SmallParams {
    RouteParams rp;          // routing inputs and outputs (the tile fields are unused)
    MoveParams mp;           // payload segments (the pipeline fields are unused)
    int n_per;               // token slots per CTA, 1..kSmallMaxTokens
    uint32_t stage_bytes;    // shared memory per token row (segments at seg_off)
    FastDiv div_tm, div_el;  // division by max_tokens and by e_local
};

struct CombineParams {
    const uint8_t *expert_out;   // [E*Ecap][h] bf16
    const int32_t *pair_row;
    const float *pair_w;
    void *out;
    int K, h, n_tokens;
    int n_rows;                  // E*Ecap: pair rows at or past it are never read
    int nvec;                    // h / 8; n_tokens * nvec < 2^31
    int groups;                  // threads per token: ceil(nvec / vectors per thread)
    FastDiv div_groups;
};

// Two-stage combine, stage 1: per received slot, the bf16-rounded fp32 sum of its
// weighted columns, into part rows [W(d)][W(s)][Tm] of part_stride bytes.
struct PartialParams {
    const uint8_t *expert_out;      // [E*Ecap][h] bf16
    const int32_t *send_cnt, *recv_eloc, *recv_row;
    const float *recv_w;
    uint8_t *part;
    size_t part_stride;
    int W, Tm, S, e_local, Ecap, h, nvec;
    uint32_t n_items;               // W*W*Tm*nvec < 2^31
    FastDiv div_nvec, div_tm, div_w;
};

// Two-stage combine, stage 2: per token, the sum over its destinations in
// ascending order of the stage-1 rows, in the output type.
struct GatherParams {
    const uint8_t *part;
    size_t part_stride;
    const int32_t *pair_send;       // [W*Tm][K] send row (s*W+d)*Tm+slot of a token's first pair on d
    void *out;
    int W, Tm, K, h, nvec;
    uint32_t n_items;               // W*Tm*nvec
    FastDiv div_nvec, div_tm;
};

// Dispatch with apply_router_weight_on_input (top_k == 1): scaled row copies.
struct ScaleMoveParams {
    const uint8_t *a1;
    const float *weights;            // [W*Tm]
    const int32_t *dst_index;        // [W*Tm] destination row of each token's pair, -1
    int n_dst_rows;                  // rows of the destination
    uint32_t a1_bytes, nvec_a1;      // 2h, 2h / 16
    int n_seg;
    const uint8_t *src_seg[kMaxSeg];  // extras (index 1..)
    uint32_t seg_vecs[kMaxSeg];       // 16-byte vectors of each extra row
    uint32_t seg_off[kMaxSeg];        // byte offset of each segment in a combined row
    uint8_t *dst[kMaxSeg];            // split: b_a1, extra_out...; combined: send_x in dst[0]
    size_t dst_stride[kMaxSeg];
    int combined;
    uint32_t vecs;                    // vectors per token (a1 + extras)
    uint32_t n_items;                 // W*Tm*vecs < 2^31
    FastDiv div_vecs;
};

struct ZeroPadParams {
    int n_seg;
    uint32_t seg_bytes[kMaxSeg];
    uint8_t *dst_seg[kMaxSeg];
    const int32_t *expert_num_tokens;   // [E]
    int E, Ecap;
    // received-slot metadata past the counts gets the page's fill values
    const int32_t *send_cnt;
    int32_t *recv_eloc, *recv_row;
    float *recv_w;
    int W, Tm, S;
};

// --------------------------------------------------------------- device utils
__device__ __forceinline__ void raise_error(DevHeader *hdr, int32_t code) {
    atomicCAS(&hdr->err, 0, code);
    atomicAdd(&hdr->err_count, 1u);
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Publishing a CTA's results: every writing thread passes a __syncthreads()
// first, then one thread stores the flag with release semantics; the release is
// cumulative, so it orders the whole CTA's earlier writes before the flag for
// any thread that reads the flag with acquire semantics.
__device__ __forceinline__ void st_release_u32(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Programmatic dependent launch: let the next kernel on the stream start its
// prologue / wait until the previous kernel's writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------ mbarrier + bulk async copies
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase; false (and an EP_ERR_TIMEOUT raise) if the
// limit runs out first.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                                  DevHeader *hdr) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > limit_ns) {
            raise_error(hdr, EP_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// global -> shared bulk copy completing on an mbarrier (bytes % 16 == 0, both
// addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// shared -> global bulk copy tracked by the bulk async-group of this thread.
__device__ __forceinline__ void bulk_s2g(void *gmem_dst, const void *smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(gmem_dst), "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until all of this thread's bulk groups have completed (writes done).
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ------------------------------------------------------------- kernel launchers
// Raise kernel fn's dynamic shared-memory limit to `bytes` on the current
// device unless that (kernel, device) already has it (see smem_limit.h).
inline cudaError_t ensure_dyn_smem(const void *fn, size_t bytes) {
    if (bytes <= SmemLimits::kDefaultLimit) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return static_cast<cudaError_t>(smem_limits().ensure(fn, dev, bytes, [&] {
        return static_cast<int>(
            cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes));
    }));
}

// Each returns the cudaError_t of the launch.
cudaError_t launch_route(const RouteParams &p, cudaStream_t st);
size_t route_smem_bytes(int n_ctr, int top_k);
cudaError_t launch_move(int mode, const MoveParams &p, int grid, int block, size_t smem, bool pdl,
                        cudaStream_t st);
// Routing and the fused row movement in one persistent launch (grid = resident CTAs).
cudaError_t launch_dispatch_fused(const RouteParams &rp, const MoveParams &mp, int grid,
                                  size_t move_smem, cudaStream_t st);
size_t small_smem_bytes(int n_per, uint32_t stage_bytes, int n_ctr, int top_k, int W, int threads);
int small_threads(int top_k);
cudaError_t launch_dispatch_small(const SmallParams &sp, int grid, int threads, size_t smem,
                                  cudaStream_t st);
cudaError_t launch_combine(const CombineParams &p, bool out_f32, int grid, bool pdl,
                           cudaStream_t st);
cudaError_t combine_occupancy(int top_k, bool out_f32, int *ctas_per_sm);
// 16-byte vectors of one token a combine thread reduces (more for small top_k,
// so that every thread keeps several loads in flight)
int combine_vectors_per_thread(int top_k);
cudaError_t launch_zero_pad(const ZeroPadParams &p, int grid_x, cudaStream_t st);
cudaError_t launch_scale_move(const ScaleMoveParams &p, int grid, cudaStream_t st);
// both stages as one-wave grids over num_sms SMs
cudaError_t launch_combine_two_stage(const PartialParams &a, const GatherParams &b, bool out_f32,
                                     int num_sms, cudaStream_t st);

}  // namespace ep
