// route.cu -- routing and slot assignment of the EP dispatch (one kernel).
//
// Computes, for all W simulated ranks at once, what `prepare` of vLLM
// AllToAllBatchedPrepareAndFinalize derives from topk_ids before any row moves:
// the destination rank of every (token, expert) pair, one slot per (rank,
// destination, token) numbered in token order, the per-destination counts
// (send_cnt), the row every pair takes inside its expert's batch (rows of an
// expert ordered by source rank, then slot), expert_num_tokens, and the
// received-slot metadata (local expert ids, router weights, rows).
//
// Both numberings are exclusive prefix counts over tokens in (rank, token)
// order: slots count, per destination d, the earlier tokens of the same rank
// that reach d; rows count, per expert e, all earlier tokens (any rank) that
// chose e. One CTA takes a tile of 256 tokens of one rank, one thread per
// token:
//   1. each warp builds lane bitmasks per destination and per expert in shared
//      memory (atomicOr of the lane bit; a token reaching a rank twice sets the
//      same bit, which deduplicates (dest, token) for free);
//   2. a block histogram turns the bitmasks into per-warp offsets and the tile
//      aggregate of every counter;
//   3. a single-pass decoupled look-back (tiles take an atomic ticket, so a tile
//      only ever waits on tiles already running) combines the aggregates and
//      inclusive prefixes of up to 32 predecessor tiles per step into the tile's
//      exclusive prefix; the destination counters restart at every rank;
//   4. each thread writes its pairs' slots, rows and metadata.
// Every wait is bounded: past the limit the tile records EP_ERR_TIMEOUT and
// finishes with what it has, so no launch can hang.
#include "ep_internal.cuh"

namespace ep {

size_t route_smem_bytes(int n_ctr) {
    // bits[warps][n_ctr] + woff[warps][n_ctr] + excl[n_ctr] + agg[n_ctr]
    return (size_t)(2 * kRouteWarps + 2) * (size_t)n_ctr * sizeof(uint32_t);
}

// Wait until tile flag f shows this launch's epoch with a published state
// (1 = aggregate, 2 = inclusive prefix). Returns the state, or 3 after the
// wait limit (EP_ERR_TIMEOUT raised).
__device__ __forceinline__ uint32_t wait_tile_flag(const uint32_t *f, uint32_t epoch,
                                                   uint64_t limit_ns, DevHeader *hdr) {
    uint32_t v = ld_acquire_u32(f);
    if ((v >> 2) == epoch && (v & 3u)) return v & 3u;
    const uint64_t t0 = global_ns();
    uint32_t back = 32;
    for (;;) {
        __nanosleep(back);
        if (back < 256) back <<= 1;
        v = ld_acquire_u32(f);
        if ((v >> 2) == epoch && (v & 3u)) return v & 3u;
        if (global_ns() - t0 > limit_ns) {
            raise_error(hdr, EP_ERR_TIMEOUT);
            return 3u;
        }
    }
}

__global__ void __launch_bounds__(kRouteTile) route_kernel(const RouteParams p) {
    extern __shared__ __align__(16) uint32_t sm[];
    const int n_ctr = p.n_ctr;
    uint32_t *bits = sm;                                               // [warps][n_ctr]
    int32_t *woff = reinterpret_cast<int32_t *>(sm + kRouteWarps * n_ctr);  // [warps][n_ctr]
    int32_t *excl = woff + kRouteWarps * n_ctr;                        // [n_ctr]
    int32_t *agg = excl + n_ctr;                                       // [n_ctr]
    __shared__ int s_tile, s_lo, s_found, s_bad;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        s_tile = (int)atomicAdd(&p.hdr->ticket, 1u);
        s_bad = 0;
    }
    for (int i = tid; i < kRouteWarps * n_ctr; i += kRouteTile) bits[i] = 0u;
    for (int i = tid; i < n_ctr; i += kRouteTile) excl[i] = 0;
    __syncthreads();
    // Every routing CTA is resident once it gets here, so the row mover may
    // launch: it cannot starve a routing tile of an SM.
    pdl_launch_dependents();

    const int q = s_tile;
    if (q >= p.num_tiles) {   // a stale ticket counter; never expected
        if (tid == 0) raise_error(p.hdr, EP_ERR_STATE);
        return;
    }
    const int W = p.W, K = p.K, e_local = p.e_local;
    const int s = q / p.tiles_per_rank;
    const int t = (q - s * p.tiles_per_rank) * kRouteTile + tid;
    int T = p.num_tokens ? p.num_tokens[s] : p.Tm;
    if (T < 0 || T > p.Tm) {
        if (tid == 0 && q % p.tiles_per_rank == 0) raise_error(p.hdr, EP_ERR_CAPACITY);
        T = T < 0 ? 0 : p.Tm;
    }
    const bool has_row = t < p.Tm;   // thread maps to a token row of the layout
    const bool valid = t < T;        // ... and that token takes part
    const int64_t g = (int64_t)s * p.Tm + t;

    // 1. the token's pairs, validated, and the lane bitmasks
    int ek[EP_MAX_TOPK], dk[EP_MAX_TOPK];
    float wk[EP_MAX_TOPK];
    uint32_t keep = 0;
#pragma unroll
    for (int k = 0; k < EP_MAX_TOPK; ++k) {
        ek[k] = -1;
        dk[k] = -1;
        wk[k] = 0.f;
        if (k < K && valid) {
            ek[k] = p.ids[g * K + k];
            wk[k] = p.weights[g * K + k];
        }
    }
#pragma unroll
    for (int k = 0; k < EP_MAX_TOPK; ++k) {
        const int e = ek[k];
        if (k >= K || !valid || e < 0) continue;
        if (e >= p.E) {
            raise_error(p.hdr, EP_ERR_EXPERT_ID);
            continue;
        }
        bool dup = false;
#pragma unroll
        for (int k2 = 0; k2 < k; ++k2) dup |= ((keep >> k2) & 1u) && ek[k2] == e;
        if (dup) {
            raise_error(p.hdr, EP_ERR_DUPLICATE);
            continue;
        }
        keep |= 1u << k;
        dk[k] = e / e_local;
        atomicOr(&bits[warp * n_ctr + dk[k]], 1u << lane);
        atomicOr(&bits[warp * n_ctr + W + e], 1u << lane);
    }
    __syncthreads();

    // 2. block histogram: per-warp exclusive offsets and the tile aggregate
    for (int c = tid; c < n_ctr; c += kRouteTile) {
        int run = 0;
#pragma unroll
        for (int w2 = 0; w2 < kRouteWarps; ++w2) {
            woff[w2 * n_ctr + c] = run;
            run += __popc(bits[w2 * n_ctr + c]);
        }
        agg[c] = run;
    }
    __syncthreads();

    // 3. decoupled look-back over the tiles before this one
    const size_t vec = (size_t)n_ctr;
    const bool publish = q != p.fault_skip_tile;
    if (q > 0) {
        for (int c = tid; c < n_ctr; c += kRouteTile) p.tile_agg[(size_t)q * vec + c] = agg[c];
        __syncthreads();
        if (tid == 0 && publish) {
            __threadfence();
            st_release_u32(&p.tile_flag[q], (p.epoch << 2) | 1u);
        }
        int pidx = q - 1;
        for (;;) {
            if (warp == 0) {
                const int idx = pidx - lane;
                uint32_t st = 0;
                if (idx >= 0) st = wait_tile_flag(&p.tile_flag[idx], p.epoch, p.wait_limit_ns, p.hdr);
                const uint32_t inc = __ballot_sync(0xffffffffu, idx >= 0 && st >= 2u);
                if (__any_sync(0xffffffffu, st == 3u) && lane == 0) s_bad = 1;
                if (lane == 0) {
                    if (inc) {
                        s_lo = pidx - (__ffs(inc) - 1);   // nearest tile with a prefix
                        s_found = 1;
                    } else {
                        s_lo = pidx - 31 > 0 ? pidx - 31 : 0;
                        s_found = 0;
                    }
                }
            }
            __syncthreads();
            const int lo = s_lo, found = s_found;
            const int rank_lo = s * p.tiles_per_rank;   // slot counters restart at each rank
            for (int c = tid; c < n_ctr; c += kRouteTile) {
                const int from = c < W ? max(lo, rank_lo) : lo;
                int v = 0;
                // independent loads (no early exit), so they are in flight together
#pragma unroll 8
                for (int idx = from; idx <= pidx; ++idx) {
                    const int32_t *src = (found && idx == lo) ? p.tile_incl : p.tile_agg;
                    v += __ldcg(src + (size_t)idx * vec + c);
                }
                excl[c] += v;
            }
            if (found || lo == 0) break;   // uniform: both read from shared memory
            pidx = lo - 1;
            __syncthreads();
        }
    }
    for (int c = tid; c < n_ctr; c += kRouteTile) p.tile_incl[(size_t)q * vec + c] = excl[c] + agg[c];
    __syncthreads();
    if (tid == 0 && publish) {
        __threadfence();
        st_release_u32(&p.tile_flag[q], (p.epoch << 2) | 2u);
    }

    // 4. per-pair outputs. After a timed-out wait the prefix is not trusted:
    // the tile marks its pairs as taking no part. Every index is range-checked
    // before it is used, so a bad prefix can never write out of bounds.
    const bool bad = s_bad != 0;
    if (has_row) {
        const uint32_t lt = lanemask_lt();
        const uint32_t *wb = bits + warp * n_ctr;
        const int32_t *wo = woff + warp * n_ctr;
#pragma unroll
        for (int k = 0; k < EP_MAX_TOPK; ++k) {
            if (k >= K) continue;
            int32_t prow = -1, psend = -1;
            float pw = 0.f;
            if (((keep >> k) & 1u) && !bad) {
                const int e = ek[k], d = dk[k], j = e - d * e_local;
                const int slot = excl[d] + wo[d] + __popc(wb[d] & lt);
                const int row = excl[W + e] + wo[W + e] + __popc(wb[W + e] & lt);
                if (slot < 0 || slot >= T || row < 0 || row >= p.Ecap) {
                    raise_error(p.hdr, EP_ERR_STATE);
                    goto store_pair;
                }
                int col = 0, n_on_d = 0;
#pragma unroll
                for (int k2 = 0; k2 < EP_MAX_TOPK; ++k2) {
                    if (k2 < K && dk[k2] == d) {
                        if (k2 < k) ++col;
                        ++n_on_d;
                    }
                }
                prow = e * p.Ecap + row;
                pw = wk[k];
                const size_t rb = ((size_t)(d * W + s) * p.Tm + slot) * p.S;
                p.recv_eloc[rb + col] = j;
                p.recv_w[rb + col] = pw;
                p.recv_row[rb + col] = row;
                if (col == 0) {
                    psend = (s * W + d) * p.Tm + slot;
                    for (int c = n_on_d; c < p.S; ++c) {
                        p.recv_eloc[rb + c] = -1;
                        p.recv_w[rb + c] = 0.f;
                        p.recv_row[rb + c] = -1;
                    }
                }
            }
        store_pair:
            p.pair_row[g * K + k] = prow;
            p.pair_w[g * K + k] = pw;
            p.pair_send[g * K + k] = psend;
        }
    }

    // per-rank slot counts and per-expert row counts
    if (q % p.tiles_per_rank == p.tiles_per_rank - 1)
        for (int c = tid; c < W; c += kRouteTile)
            p.send_cnt[s * W + c] = bad ? 0 : min(max(excl[c] + agg[c], 0), T);
    if (q == p.num_tiles - 1)
        for (int e = tid; e < p.E; e += kRouteTile)
            p.expert_num_tokens[e] = bad ? 0 : min(max(excl[W + e] + agg[W + e], 0), p.Ecap);

    // the last tile to finish rearms the ticket for the next launch
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(&p.hdr->done, 1u) == (uint32_t)p.num_tiles - 1) {
            atomicExch(&p.hdr->ticket, 0u);
            atomicExch(&p.hdr->done, 0u);
        }
    }
}

cudaError_t launch_route(const RouteParams &p, size_t smem, cudaStream_t st) {
    static size_t smem_set = 0;
    if (smem > 48 * 1024 && smem > smem_set) {
        cudaError_t e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        smem_set = smem;
    }
    route_kernel<<<p.num_tiles, kRouteTile, smem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace ep
