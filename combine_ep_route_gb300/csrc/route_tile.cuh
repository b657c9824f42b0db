// route_tile.cuh -- one tile of the routing and slot assignment of the EP
// dispatch, as a device function shared by the routing kernel and by the
// persistent dispatch kernel that routes and then moves rows in one launch.
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
// chose e. One CTA of 256 threads takes a tile of 64 tokens of one rank:
//   1. one thread per token validates its top-k ids and sets its lane bit in
//      per-warp bitmasks, one per destination and one per expert (atomicOr in
//      shared memory; a token reaching a rank twice sets the same bit, which
//      deduplicates (dest, token) for free);
//   2. a block histogram turns the bitmasks into per-warp offsets and the tile
//      aggregate of every counter;
//   3. a single-pass decoupled look-back (tiles take an atomic ticket, so a tile
//      only ever waits on tiles already running) combines the aggregates and
//      inclusive prefixes of up to 32 predecessor tiles per step into the tile's
//      exclusive prefix; the destination counters restart at every rank;
//   4. one thread per (token, k) pair writes the pair's row, weight and slot
//      (coalesced) and the tile publishes them; then the first pair of a token
//      on each destination writes that destination's received-slot row with
//      16-byte vector stores.
// Every wait is bounded: past the limit the tile records EP_ERR_TIMEOUT and
// finishes with what it has, so no launch can hang.
#pragma once

#include "ep_internal.cuh"

namespace ep {

inline int route_kt(int top_k) {
    int kt = 1;
    while (kt < top_k) kt <<= 1;
    return kt;
}

inline size_t route_smem_bytes(int n_ctr, int top_k) {
    // bits[warps][n_ctr] + woff[warps][n_ctr] + excl[n_ctr] + agg[n_ctr]
    // + the tile's kept pairs and weights [64][kt]
    return (size_t)(2 * kRouteWarps + 2) * (size_t)n_ctr * sizeof(uint32_t) +
           (size_t)kRouteTile * route_kt(top_k) * (sizeof(int32_t) + sizeof(float));
}

// Tile flag states (low two bits; the epoch is above them): 1 = aggregate
// published, 2 = inclusive prefix published, 3 = prefix and pair outputs published.
constexpr uint32_t kFlagAgg = 1u, kFlagIncl = 2u, kFlagDone = 3u;
constexpr uint32_t kFlagTimeout = 4u;   // what a wait returns when its limit runs out

// Wait until tile flag f shows this launch's epoch with a published state.
// Returns the state, or kFlagTimeout after the wait limit (EP_ERR_TIMEOUT raised).
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
            return kFlagTimeout;
        }
    }
}

// One routing tile (ticket q) with the whole CTA (kRouteThreads threads), using
// shared memory sm (route_smem_bytes). epoch: this launch's look-back epoch.
// When it returns, the tile's outputs are written, and its flag reads
// `epoch << 2 | 3` (3 = the pair outputs are published: pair_row, pair_w and
// pair_send; the received-slot rows and counts are written after it and are
// for later launches; the look-back treats 2 and 3 alike).
// KT: top_k rounded up to a power of two (compile-time loop bounds).
template <int KT>
__device__ void route_tile(const RouteParams &p, const int q, const uint32_t epoch, uint32_t *sm) {
    const int n_ctr = p.n_ctr;
    uint32_t *bits = sm;                                               // [warps][n_ctr]
    int32_t *woff = reinterpret_cast<int32_t *>(sm + kRouteWarps * n_ctr);  // [warps][n_ctr]
    int32_t *excl = woff + kRouteWarps * n_ctr;                        // [n_ctr]
    int32_t *agg = excl + n_ctr;                                       // [n_ctr]
    int32_t *sid = agg + n_ctr;   // [64][KT] kept pair: dest << 16 | expert id; -1 if dropped
    float *sw = reinterpret_cast<float *>(sid + kRouteTile * KT);      // [64][KT]
    __shared__ int s_lo, s_found, s_bad;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    __syncthreads();   // shared memory may still be in use by the caller's previous step
    if (tid == 0) s_bad = 0;
    for (int i = tid; i < kRouteWarps * n_ctr; i += kRouteThreads) bits[i] = 0u;
    for (int i = tid; i < n_ctr; i += kRouteThreads) excl[i] = 0;
    __syncthreads();

    const int W = p.W, K = p.K, e_local = p.e_local;
    const int s = q / p.tiles_per_rank;
    const int t0 = (q - s * p.tiles_per_rank) * kRouteTile;   // first token of the tile
    // the rank's token count and the tile's ids are loaded together: ids of every
    // token below max_tokens are read, and those at or past the count dropped after
    const int T_in = p.num_tokens ? __ldg(p.num_tokens + s) : p.Tm;

    // 1. one thread per token: load, validate, lane bitmasks
    int ek[KT];
    float wk[KT];
    if (tid < kRouteTile) {
        const int t = t0 + tid;
        const bool inb = t < p.Tm;
        const int64_t g = (int64_t)s * p.Tm + t;
        if (inb && KT % 4 == 0 && K == KT && p.vec_ids) {
            const int4 *pi = reinterpret_cast<const int4 *>(p.ids + g * KT);
            const float4 *pw = reinterpret_cast<const float4 *>(p.weights + g * KT);
#pragma unroll
            for (int v = 0; v < KT / 4; ++v) {
                const int4 a = __ldg(pi + v);
                const float4 b = __ldg(pw + v);
                ek[4 * v] = a.x, ek[4 * v + 1] = a.y, ek[4 * v + 2] = a.z, ek[4 * v + 3] = a.w;
                wk[4 * v] = b.x, wk[4 * v + 1] = b.y, wk[4 * v + 2] = b.z, wk[4 * v + 3] = b.w;
            }
        } else {
#pragma unroll
            for (int k = 0; k < KT; ++k) {
                ek[k] = (inb && k < K) ? __ldg(p.ids + g * K + k) : -1;
                wk[k] = (inb && k < K) ? __ldg(p.weights + g * K + k) : 0.f;
            }
        }
    }
    int T = T_in;
    if (T < 0 || T > p.Tm) {
        if (tid == 0 && q % p.tiles_per_rank == 0) raise_error(p.hdr, EP_ERR_CAPACITY);
        T = T < 0 ? 0 : p.Tm;
    }
    if (tid < kRouteTile) {
        if (t0 + tid >= T) {
#pragma unroll
            for (int k = 0; k < KT; ++k) ek[k] = -1;
        }
        uint32_t keep = 0;
#pragma unroll
        for (int k = 0; k < KT; ++k) {
            const int e = ek[k];
            bool ok = k < K && e >= 0;
            if (ok && e >= p.E) {
                raise_error(p.hdr, EP_ERR_EXPERT_ID);
                ok = false;
            }
            if (ok) {
                bool dup = false;
#pragma unroll
                for (int k2 = 0; k2 < k; ++k2) dup |= ((keep >> k2) & 1u) && ek[k2] == e;
                if (dup) {
                    raise_error(p.hdr, EP_ERR_DUPLICATE);
                    ok = false;
                }
            }
            int packed = -1;
            if (ok) {
                const int d = e / e_local;
                keep |= 1u << k;
                atomicOr(&bits[warp * n_ctr + d], 1u << lane);
                atomicOr(&bits[warp * n_ctr + W + e], 1u << lane);
                packed = (d << 16) | e;   // e < 2^16, d < 2^15 (EP_MAX_E, EP_MAX_W)
            }
            sid[tid * KT + k] = packed;
            sw[tid * KT + k] = wk[k];
        }
    }
    __syncthreads();

    // 2. block histogram: per-warp exclusive offsets and the tile aggregate
    for (int c = tid; c < n_ctr; c += kRouteThreads) {
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
        for (int c = tid; c < n_ctr; c += kRouteThreads) p.tile_agg[(size_t)q * vec + c] = agg[c];
        __syncthreads();
        if (tid == 0 && publish) {
            st_release_u32(&p.tile_flag[(size_t)q * kFlagStride], (epoch << 2) | kFlagAgg);
        }
        int pidx = q - 1;
        for (;;) {
            if (warp == 0) {
                const int idx = pidx - lane;
                uint32_t st = 0;
                if (idx >= 0)
                    st = wait_tile_flag(&p.tile_flag[(size_t)idx * kFlagStride], epoch, p.wait_limit_ns, p.hdr);
                // a prefix (or a timed-out wait, whose tile is then marked bad) ends the walk
                const uint32_t inc = __ballot_sync(0xffffffffu, idx >= 0 && st >= kFlagIncl);
                if (__any_sync(0xffffffffu, st == kFlagTimeout) && lane == 0) s_bad = 1;
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
            for (int c = tid; c < n_ctr; c += kRouteThreads) {
                const int from = c < W ? max(lo, rank_lo) : lo;
                // the window is at most 32 tiles: issue every load before the first add
                int part[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int idx = pidx - i;
                    part[i] = 0;
                    if (idx >= from) {
                        const int32_t *src = (found && idx == lo) ? p.tile_incl : p.tile_agg;
                        part[i] = __ldcg(src + (size_t)idx * vec + c);
                    }
                }
                int v = 0;
#pragma unroll
                for (int i = 0; i < 32; ++i) v += part[i];
                excl[c] += v;
            }
            if (found || lo == 0) break;   // uniform: both read from shared memory
            pidx = lo - 1;
            __syncthreads();
        }
    }
    for (int c = tid; c < n_ctr; c += kRouteThreads) p.tile_incl[(size_t)q * vec + c] = excl[c] + agg[c];
    __syncthreads();
    if (tid == 0 && publish) st_release_u32(&p.tile_flag[(size_t)q * kFlagStride], (epoch << 2) | kFlagIncl);

    // 4. one thread per (token, k) pair. (a) Each pair's row, weight and send
    // slot are written (coalesced) and published: that is all the row movers of
    // the same launch read. (b) Then the first pair of a token on each
    // destination writes that destination's whole received-slot row (S columns
    // of local id, weight and row), assembled in registers and stored as
    // 16-byte vectors, and the tile's last counters are written; later
    // launches read those. After a timed-out wait the prefix is not trusted:
    // the tile marks its pairs as taking no part. Every index is range-checked
    // before it is used, so a bad prefix can never write out of bounds.
    const bool bad = s_bad != 0;
    const int rows_in_tile = min(kRouteTile, p.Tm - t0);
    // slot of the pair's token on destination d and the pair's row in its
    // expert; false if the pair was dropped or its position is out of range
    auto locate = [&](int tl, int pk, int &slot, int &row) -> bool {
        if (pk < 0 || bad) return false;
        const int e = pk & 0xFFFF, d = pk >> 16;
        const int tw = tl >> 5;
        const uint32_t lt = (1u << (tl & 31)) - 1u;
        const uint32_t *wb = bits + tw * n_ctr;
        const int32_t *wo = woff + tw * n_ctr;
        slot = excl[d] + wo[d] + __popc(wb[d] & lt);
        row = excl[W + e] + wo[W + e] + __popc(wb[W + e] & lt);
        return slot >= 0 && slot < T && row >= 0 && row < p.Ecap;
    };
    // true if no earlier kept pair of the token goes to the same destination
    auto first_on_dest = [&](const int32_t *te, int k, int d) -> bool {
        bool first = true;
#pragma unroll
        for (int k2 = 0; k2 < KT; ++k2)
            if (k2 < k && te[k2] >= 0 && (te[k2] >> 16) == d) first = false;
        return first;
    };
    for (int pi = tid; pi < rows_in_tile * KT; pi += kRouteThreads) {
        const int tl = pi / KT, k = pi % KT;
        if (k >= K) continue;
        const int64_t g = (int64_t)s * p.Tm + t0 + tl;
        const int32_t *te = sid + tl * KT;
        const int pk = te[k];
        int32_t prow = -1, psend = -1;
        float pw = 0.f;
        int slot = 0, row = 0;
        if (locate(tl, pk, slot, row)) {
            const int e = pk & 0xFFFF, d = pk >> 16;
            prow = e * p.Ecap + row;
            pw = p.unit_weights ? 1.0f : sw[tl * KT + k];
            if (first_on_dest(te, k, d)) psend = (s * W + d) * p.Tm + slot;
        } else if (pk >= 0 && !bad) {
            raise_error(p.hdr, EP_ERR_STATE);
        }
        p.pair_row[g * K + k] = prow;
        p.pair_w[g * K + k] = pw;
        p.pair_send[g * K + k] = psend;
    }
    __syncthreads();
    if (tid == 0 && publish) st_release_u32(&p.tile_flag[(size_t)q * kFlagStride], (epoch << 2) | kFlagDone);

    for (int pi = tid; pi < rows_in_tile * KT; pi += kRouteThreads) {
        const int tl = pi / KT, k = pi % KT;
        if (k >= K) continue;
        const int32_t *te = sid + tl * KT;
        const int pk = te[k];
        int slot = 0, row = 0;
        if (!locate(tl, pk, slot, row)) continue;
        const int d = pk >> 16;
        if (!first_on_dest(te, k, d)) continue;
        // columns: the token's pairs on d in top-k order, then unused
        const int tw = tl >> 5;
        const uint32_t lt = (1u << (tl & 31)) - 1u;
        const uint32_t *wb = bits + tw * n_ctr;
        const int32_t *wo = woff + tw * n_ctr;
        int cj[KT], cr[KT];
        float cw[KT];
#pragma unroll
        for (int c = 0; c < KT; ++c) {
            cj[c] = -1;
            cr[c] = -1;
            cw[c] = 0.f;
        }
        int n = 0;
        const int jbase = d * e_local;
#pragma unroll
        for (int k2 = 0; k2 < KT; ++k2) {
            const int p2 = te[k2];
            if (p2 >= 0 && (p2 >> 16) == d) {
                const int e2 = p2 & 0xFFFF;
                const int r2 = excl[W + e2] + wo[W + e2] + __popc(wb[W + e2] & lt);
                const float w2 = p.unit_weights ? 1.0f : sw[tl * KT + k2];
#pragma unroll
                for (int c = 0; c < KT; ++c)
                    if (c == n) {
                        cj[c] = e2 - jbase;
                        cr[c] = r2;
                        cw[c] = w2;
                    }
                ++n;
            }
        }
        const size_t rb = ((size_t)(d * W + s) * p.Tm + slot) * p.S;
        if (KT >= 4 && p.vec_recv) {   // S % 4 == 0, 16-byte aligned rows
#pragma unroll
            for (int c4 = 0; c4 < KT / 4; ++c4) {
                if (4 * c4 >= p.S) break;
                reinterpret_cast<int4 *>(p.recv_eloc + rb)[c4] =
                    make_int4(cj[4 * c4], cj[4 * c4 + 1], cj[4 * c4 + 2], cj[4 * c4 + 3]);
                reinterpret_cast<int4 *>(p.recv_row + rb)[c4] =
                    make_int4(cr[4 * c4], cr[4 * c4 + 1], cr[4 * c4 + 2], cr[4 * c4 + 3]);
                reinterpret_cast<float4 *>(p.recv_w + rb)[c4] =
                    make_float4(cw[4 * c4], cw[4 * c4 + 1], cw[4 * c4 + 2], cw[4 * c4 + 3]);
            }
        } else {
#pragma unroll
            for (int c = 0; c < KT; ++c) {
                if (c >= p.S) break;
                p.recv_eloc[rb + c] = cj[c];
                p.recv_row[rb + c] = cr[c];
                p.recv_w[rb + c] = cw[c];
            }
        }
    }

    // per-rank slot counts and per-expert row counts
    if (q % p.tiles_per_rank == p.tiles_per_rank - 1)
        for (int c = tid; c < W; c += kRouteThreads)
            p.send_cnt[s * W + c] = bad ? 0 : min(max(excl[c] + agg[c], 0), T);
    if (q == p.num_tiles - 1)
        for (int e = tid; e < p.E; e += kRouteThreads)
            p.expert_num_tokens[e] = bad ? 0 : min(max(excl[W + e] + agg[W + e], 0), p.Ecap);
}

}  // namespace ep
