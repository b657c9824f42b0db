// move.cu -- the row movement of the EP dispatch, as bulk asynchronous copies.
//
// All four row-moving steps of `prepare` (vLLM AllToAllBatchedPrepareAndFinalize)
// have one shape: read a row (an a1 row, possibly followed by extra payload
// rows) once and write it to a handful of destination rows. One kernel
// template serves them:
//   MOVE_FUSED    a1[s][t] (+ extras)  -> b_a1[d][j][row] of every pair of t
//                 (the direct path: no send or receive buffers)
//   MOVE_PACK     a1[s][t] (+ extras)  -> send_x[s][d][slot] of every rank t reaches
//   MOVE_EXCHANGE send_x[s][d][slot]   -> recv_x[d][s][slot]  (the all_to_all_single
//                 of a multi-GPU run, here a permutation of rank blocks in HBM)
//   MOVE_DELIVER  recv_x[d][s][slot]   -> b_a1[d][j][row] (+ extras) of every column
//
// Each warp of a CTA runs its own pipeline over a ring of shared-memory stages:
// lane 0 loads a unit's row into a stage with cp.async.bulk (completion on an
// mbarrier), then stores it to every destination with cp.async.bulk from
// shared memory; the stage is refilled once the bulk group that read it is done.
// The other lanes fetch the next unit's destination list while the current
// unit's copies are in flight. Rows never pass through registers, and a row
// with k destinations is read from HBM once. A unit is one chunk of a row's
// activation part (the extra payloads travel with chunk 0): many equal units
// per pipeline keep the tail of the persistent grid short.
#include "route_tile.cuh"

namespace ep {

namespace {

// An L2 evict-first policy for the mover's source reads. Every source row (or
// chunk of one) is read once, so it need not stay in L2, where it would displace
// the destination rows the combine reads next (measured on GB300: prefill step
// -0.5 us, Zipf -0.8 us, grouped -0.7 us; the same hint on the stores instead
// made the combine 2.5-5 us slower).
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// global -> shared bulk copy (completion on an mbarrier) with an L2 cache policy
__device__ __forceinline__ void bulk_g2s_hint(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                              uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// Wait (bounded) until a routing tile of this launch has published its
// outputs. False after the limit (EP_ERR_TIMEOUT raised).
__device__ __forceinline__ bool wait_tile_done(const uint32_t *f, uint32_t epoch, uint64_t limit_ns,
                                               DevHeader *hdr) {
    const uint32_t want = (epoch << 2) | kFlagDone;
    if (ld_acquire_u32(f) == want) return true;
    const uint64_t t0 = global_ns();
    uint32_t back = 64;
    for (;;) {
        __nanosleep(back);
        if (back < 1024) back <<= 1;
        if (ld_acquire_u32(f) == want) return true;
        if (global_ns() - t0 > limit_ns) {
            raise_error(hdr, EP_ERR_TIMEOUT);
            return false;
        }
    }
}

// How long a mover's launch-time stage fills wait, at most, for their routing
// tile to publish anything (move_body).
constexpr uint64_t kFillWaitNs = 20000;

// Largest b in [0, nb) with pre[b] <= u, for pre[0] = 0 <= u < pre[nb].
__device__ __forceinline__ int find_block(const int32_t *pre, int nb, int u) {
    int lo = 0, hi = nb;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= u) lo = mid;
        else hi = mid;
    }
    return lo;
}

// Source row index (the whole warp gets it) and this lane's destination row
// index (-1 for none) of unit u.
template <int MODE>
__device__ __forceinline__ void unit_meta(const MoveParams &p, const int32_t *pre, int u, int lane,
                                          uint32_t epoch, int &src, int &dst) {
    dst = -1;
    if (MODE == MOVE_FUSED || MODE == MOVE_PACK) {
        src = u;
        if (p.wait_tiles) {
            // routing runs in this launch: wait (bounded) until the token's tile
            // has published its outputs, then read them past the L1
            const uint32_t s = fastdiv((uint32_t)u, p.div_tm);
            const int t = u - (int)s * p.Tm;
            const uint32_t *flag =
                p.tile_flag + (size_t)((int)s * p.tiles_per_rank + t / kRouteTile) * kFlagStride;
            bool ready = true;
            if (lane == 0) ready = wait_tile_done(flag, epoch, p.wait_limit_ns, p.hdr);
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (ready && lane < p.K) {
                (void)ld_acquire_u32(flag);   // each reading lane acquires the tile's release
                dst = __ldcg((MODE == MOVE_FUSED ? p.pair_row : p.pair_send) + (size_t)u * p.K + lane);
                const int lim = MODE == MOVE_FUSED ? p.n_rows : p.n_slots;
                if (dst >= lim) {
                    raise_error(p.hdr, EP_ERR_STATE);
                    dst = -1;
                }
            }
            return;
        }
        if (lane < p.K) {
            dst = (MODE == MOVE_FUSED ? p.pair_row : p.pair_send)[(size_t)u * p.K + lane];
            const int lim = MODE == MOVE_FUSED ? p.n_rows : p.n_slots;
            if (dst >= lim) {   // never produced by routing; kept out of bounds checks' way
                raise_error(p.hdr, EP_ERR_STATE);
                dst = -1;
            }
        }
    } else {
        const int W = p.W;
        const int b = find_block(pre, W * W, u);
        const int slot = u - pre[b];
        const int a = b / W, c = b - a * W;
        if (MODE == MOVE_EXCHANGE) {   // b = (s, d): send row -> recv row
            src = (a * W + c) * p.Tm + slot;
            if (lane == 0) dst = (c * W + a) * p.Tm + slot;
        } else {                       // b = (d, s): recv row -> expert rows
            src = (a * W + c) * p.Tm + slot;
            if (lane < p.S) {
                const int j = p.recv_eloc[(size_t)src * p.S + lane];
                const int r = p.recv_row[(size_t)src * p.S + lane];
                if (j >= 0) {
                    if (j < p.e_local && r >= 0 && r < p.Ecap) {
                        dst = (a * p.e_local + j) * p.Ecap + r;
                    } else {
                        raise_error(p.hdr, EP_ERR_STATE);
                    }
                }
            }
        }
    }
}

}  // namespace

// The mover's pipelines over one CTA's share of the units (see the top of the file).
template <int MODE>
__device__ __forceinline__ void move_body(const MoveParams &p, uint8_t *smem, uint32_t epoch) {
    constexpr int kStash = kMaxDst + 3;   // per stage: src, count, destinations, chunk
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int P = p.pipes;
    const uint64_t pol = evict_first_policy();   // source reads
    const int NS = p.stages;
    const size_t stage_region = (size_t)P * NS * p.stage_bytes;
    uint8_t *stages = smem + (size_t)warp * NS * p.stage_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + stage_region) + warp * NS;
    int32_t *stash = reinterpret_cast<int32_t *>(reinterpret_cast<uint64_t *>(smem + stage_region) +
                                                 P * NS) + warp * NS * kStash;
    int32_t *pre = reinterpret_cast<int32_t *>(reinterpret_cast<uint64_t *>(smem + stage_region) +
                                               P * NS) + P * NS * kStash;

    if (lane == 0) {
        for (int i = 0; i < NS; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    // Everything below reads what the previous kernel on the stream wrote.
    pdl_wait();

    int n_units;
    if (MODE == MOVE_EXCHANGE || MODE == MOVE_DELIVER) {
        // exclusive prefix of the (s, d) or (d, s) slot counts, in shared memory
        const int W = p.W, nb = W * W;
        for (int b = threadIdx.x; b < nb; b += blockDim.x) {
            const int a = b / W, c = b - a * W;
            const int n = MODE == MOVE_EXCHANGE ? p.send_cnt[b] : p.send_cnt[c * W + a];
            pre[b] = min(max(n, 0), p.Tm);   // counts are in range; the clamp keeps it so
        }
        __syncthreads();
        if (warp == 0) {
            const int per = (nb + 31) / 32;
            const int lo = lane * per, hi = min(nb, lo + per);
            int sum = 0;
            for (int b = lo; b < hi; ++b) sum += pre[b];
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            int run = incl - sum;
            for (int b = lo; b < hi; ++b) {
                const int v = pre[b];
                pre[b] = run;
                run += v;
            }
            if (lane == 31) pre[nb] = incl;
        }
        __syncthreads();
        n_units = pre[nb];
    } else {
        n_units = p.n_tokens;
        __syncwarp();
    }

    const bool src_split = MODE == MOVE_FUSED || MODE == MOVE_PACK;
    const bool dst_split = MODE == MOVE_FUSED || MODE == MOVE_DELIVER;
    const uint8_t *src_whole = MODE == MOVE_EXCHANGE ? p.send_x : p.recv_x;
    uint8_t *dst_whole = MODE == MOVE_PACK ? p.send_x : p.recv_x;

    // units = row units x chunks, chunk-minor
    const int C = p.chunks;
    const uint32_t cb = p.chunk_bytes;
    const uint32_t a1b = p.seg_bytes[0];
    const uint32_t tail = p.row_bytes - a1b;   // extra payload bytes, moved with chunk 0
    const int n_work = n_units * C;
    const int first = blockIdx.x * P + warp, stride = gridDim.x * P;

    // The warp's i-th unit: a fixed stride (static), or -- dynamic -- its first
    // kStaticUnits units by stride and the rest in batches of kUnitBatch grabbed
    // from a launch-wide counter, so a warp that starts late (after routing a
    // tile in the same launch) takes fewer units, while small problems never
    // touch the counter. The last two rounds are grabbed one unit at a time, so
    // the warps finish within about one unit of each other. Called with i
    // growing by at most one per new value. One static unit per warp, batches of
    // four and two single-unit rounds measured best on GB300 (prefill dispatch
    // 173.4 -> 172.9 us, Zipf 109.6 -> 109.1, grouped 150.9 -> 150.5; two static
    // units, batches of 2, 3, 6 or 8 and one, three or four final rounds were
    // slower).
    // (kStaticUnits must stay at least 1: the fills below read unit_at(0) once
    // before they take their units, which must not consume a dynamic batch.)
    constexpr int kStaticUnits = 1, kUnitBatch = 4;
    const bool dyn = p.dynamic_units != 0;
    const int tail_from = n_work - 2 * kUnitBatch * stride;
    int seq_base = 0, seq_len = 0, seq_i0 = kStaticUnits;
    auto unit_at = [&](int i) -> int {
        if (!dyn || i < kStaticUnits) {
            const int u = first + i * stride;
            return u < n_work ? u : -1;
        }
        while (i >= seq_i0 + seq_len) {
            if (seq_len < 0) return -1;   // the counter ran out
            // seq_base (the warp's last batch) stands in for the counter
            const int want = seq_base >= tail_from ? 1 : kUnitBatch;
            int b = 0;
            if (lane == 0) b = (int)atomicAdd(&p.hdr->move_next, (uint32_t)want);
            b = __shfl_sync(0xffffffffu, b, 0) + kStaticUnits * stride;
            seq_i0 += seq_len;
            if (b >= n_work) {
                seq_len = -1;
                return -1;
            }
            seq_base = b;
            seq_len = min(want, n_work - b);
        }
        return seq_base + (i - seq_i0);
    };

    int nxt_u = -1;
    int nxt_src = -1, nxt_dst = -1;   // metadata of the next unit to load

    // lane 0: load source row src, chunk c, into stage st (completion on its mbarrier)
    auto load_unit = [&](int st, int src, int c) {
        uint64_t *bar = &bars[st];
        uint8_t *stg = stages + (size_t)st * p.stage_bytes;
        mbar_arrive_expect_tx(bar, cb + (c == 0 ? tail : 0u));
        if (src_split) {
            bulk_g2s_hint(stg, p.src_seg[0] + (size_t)src * a1b + (size_t)c * cb, cb, bar, pol);
            if (c == 0)
                for (int sg = 1; sg < p.n_seg; ++sg)
                    bulk_g2s_hint(stg + cb + (p.seg_off[sg] - a1b),
                                  p.src_seg[sg] + (size_t)src * p.seg_bytes[sg], p.seg_bytes[sg], bar, pol);
        } else {
            const uint8_t *row = src_whole + (size_t)src * p.row_bytes;
            bulk_g2s_hint(stg, row + (size_t)c * cb, cb, bar, pol);
            if (c == 0 && tail) bulk_g2s_hint(stg + cb, row + a1b, tail, bar, pol);
        }
    };

    // Load the warp's unit i (the next one in order) into stage i % NS, then
    // fetch the metadata of unit i + 1 while that load is in flight (the fetch
    // is one or more L2 round trips: a tile flag, the token's pair rows, and in
    // the dynamic case the unit counter). Chunks of one token share metadata,
    // so it is fetched once per token.
    auto issue = [&](int i) {
        const int st = i % NS;
        int32_t *sh = stash + st * kStash;
        const bool has = nxt_dst >= 0;
        const uint32_t m = __ballot_sync(0xffffffffu, has);
        if (has) sh[2 + __popc(m & lanemask_lt())] = nxt_dst;
        const int src = nxt_src;
        const int row_unit = nxt_u / C;
        const int c = nxt_u - row_unit * C;
        if (lane == 0) {
            sh[kMaxDst + 2] = c;
            sh[0] = m ? src : -1;
            sh[1] = __popc(m);
            if (m) load_unit(st, src, c);
            else mbar_arrive(&bars[st]);   // empty unit: complete the phase with no transfer
        }
        nxt_u = unit_at(i + 1);
        if (nxt_u >= 0 && nxt_u / C != row_unit)
            unit_meta<MODE>(p, pre, nxt_u / C, lane, epoch, nxt_src, nxt_dst);
        __syncwarp();
    };

    int issued = 0;
    if (src_split && p.wait_tiles) {
        // Routing runs in this launch: fill the first stages before the
        // destinations are known. A unit's source row follows from its index,
        // so its load overlaps the wait for its routing tile; a unit that turns
        // out to have no destination was loaded for nothing and is skipped.
        // The fills wait until the first unit's tile has published anything
        // (its aggregate, ~3.5 us into a prefill launch): before that the
        // routing tiles' own loads and flag round trips are on the critical
        // path and the fills would only compete with them (measured on GB300:
        // dispatch 0.2-0.75 us faster on the prefill, Zipf and grouped
        // workloads). The wait is bounded and raises nothing: a tile that never
        // publishes is reported by the waits for its outputs.
        {
            const int u0 = unit_at(0);
            if (u0 >= 0 && lane == 0) {
                const int tok = u0 / C;
                const uint32_t s0 = fastdiv((uint32_t)tok, p.div_tm);
                const int t0 = tok - (int)s0 * p.Tm;
                const uint32_t *f0 =
                    p.tile_flag + (size_t)((int)s0 * p.tiles_per_rank + t0 / kRouteTile) * kFlagStride;
                const uint64_t start = global_ns();
                for (;;) {
                    const uint32_t v = ld_relaxed_u32(f0);
                    if ((v >> 2) == epoch && (v & 3u) != 0u) break;
                    if (global_ns() - start > kFillWaitNs) break;
                    __nanosleep(256);
                }
            }
            __syncwarp();
        }
        for (; issued < NS; ++issued) {
            const int u = unit_at(issued);
            if (u < 0) break;
            if (lane == 0) {
                int32_t *sh = stash + issued * kStash;
                const int row_unit = u / C, c = u - row_unit * C;
                sh[0] = row_unit;
                sh[kMaxDst + 2] = c;
                load_unit(issued, row_unit, c);
            }
        }
        __syncwarp();
        int prev = -1, src = -1, dst = -1;
        for (int j = 0; j < issued; ++j) {
            int32_t *sh = stash + j * kStash;
            const int row_unit = sh[0];
            __syncwarp();   // every lane has read sh[0] before lane 0 rewrites it
            if (row_unit != prev) {
                unit_meta<MODE>(p, pre, row_unit, lane, epoch, src, dst);
                prev = row_unit;
            }
            const bool has = dst >= 0;
            const uint32_t m = __ballot_sync(0xffffffffu, has);
            if (has) sh[2 + __popc(m & lanemask_lt())] = dst;
            if (lane == 0) {
                sh[0] = m ? src : -1;
                sh[1] = __popc(m);
            }
        }
        nxt_u = unit_at(issued);
        if (nxt_u >= 0) {
            if (nxt_u / C == prev) {
                nxt_src = src;
                nxt_dst = dst;
            } else {
                unit_meta<MODE>(p, pre, nxt_u / C, lane, epoch, nxt_src, nxt_dst);
            }
        }
        __syncwarp();
    } else {
        nxt_u = unit_at(0);
        if (nxt_u >= 0) unit_meta<MODE>(p, pre, nxt_u / C, lane, epoch, nxt_src, nxt_dst);
    }
    while (issued < NS && nxt_u >= 0) issue(issued++);
    int consumed = 0;
    const int last_from = n_work - 2 * stride;   // the last two rounds of units
    bool ok = true;
    for (int i = 0; i < issued; ++i) {
        const int st = i % NS;
        if (lane == 0) {
            ok = mbar_wait_bounded(&bars[st], (uint32_t)(i / NS) & 1u, p.wait_limit_ns, p.hdr);
            const int32_t *sh = stash + st * kStash;
            if (ok && sh[0] >= 0) {
                const uint8_t *stg = stages + (size_t)st * p.stage_bytes;
                const int c = sh[kMaxDst + 2];
                const int n = sh[1];
                for (int q = 0; q < n; ++q) {
                    const size_t drow = (size_t)sh[2 + q];
                    if (dst_split) {
                        bulk_s2g(p.dst_seg[0] + drow * a1b + (size_t)c * cb, stg, cb);
                        if (c == 0)
                            for (int sg = 1; sg < p.n_seg; ++sg)
                                bulk_s2g(p.dst_seg[sg] + drow * p.seg_bytes[sg],
                                         stg + cb + (p.seg_off[sg] - a1b), p.seg_bytes[sg]);
                    } else {
                        uint8_t *row = dst_whole + drow * p.row_bytes;
                        bulk_s2g(row + (size_t)c * cb, stg, cb);
                        if (c == 0 && tail) bulk_s2g(row + a1b, stg + cb, tail);
                    }
                }
            }
            bulk_commit();
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        consumed = i + 1;
        // Refill a free stage (the one unit i-1 used, or an earlier one) with
        // the next unit, if there is one. In the last two rounds of units a warp
        // loads a unit only when none of its loaded units is still waiting for
        // its stores, so the last units are spread over the warps that are
        // ready for them and the warps finish closer together (measured on
        // GB300: Zipf dispatch -0.7 us, grouped -0.45 us, prefill unchanged;
        // allowing two waiting units, or limiting one to eight rounds, gained
        // less).
        if (i >= 1 && issued <= i - 1 + NS && nxt_u >= 0 && (nxt_u < last_from || issued == i + 1)) {
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
            issue(issued++);
        }
    }
    if (lane == 0) {
        if (!ok) {
            // drain the loads already issued before leaving (bounded), the one
            // whose wait ran out included
            for (int i = consumed; i < issued; ++i)
                if (!mbar_wait_bounded(&bars[i % NS], (uint32_t)(i / NS) & 1u, p.wait_limit_ns, p.hdr))
                    break;
        }
        bulk_wait_all();
    }
}

template <int MODE>
__global__ void __launch_bounds__(256) move_kernel(const MoveParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    move_body<MODE>(p, smem, 0u);
}

// Routing and the fused row movement in one persistent launch. The first
// rp.route_ctas CTAs to arrive (all of them when it is 0) are routers: they
// take routing tiles by ticket until none is left, then join the others in
// moving rows with their first mp.pipes warps (the rest are done). A unit
// waits only for its own token's tile, so movement starts as soon as the first
// tiles are out, and routers that work through the tiles in ticket order stay
// ahead of the movers, which take tokens in roughly ascending order. No
// deadlock: every tile is routed by a router, a router is running from the
// moment it is elected, routers never wait on movers, and a tile waits only on
// tiles with smaller tickets. The last CTA to finish rearms the counters and
// advances the look-back epoch, as the routing kernel does.
template <int KT>
__global__ void __launch_bounds__(256, 2) dispatch_fused_kernel(const RouteParams rp, const MoveParams mp) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_q;
    __shared__ uint32_t s_epoch;
    const int tid = threadIdx.x;
    if (tid == 0) {
        // The epoch was last written by the previous launch (ordered before this
        // one by the launch boundary) and is written in this one only after every
        // CTA has read it: a relaxed load suffices, and the first ticket need not
        // wait for it.
        const uint32_t e = ld_relaxed_u32(&rp.hdr->epoch);
        const bool router = rp.route_ctas <= 0 || (int)atomicAdd(&rp.hdr->routers, 1u) < rp.route_ctas;
        s_q = router ? (int)atomicAdd(&rp.hdr->ticket, 1u) : rp.num_tiles;
        s_epoch = e & 0x3FFFFFFFu;
    }
    __syncthreads();
    const uint32_t epoch = s_epoch;
    for (;;) {
        const int q = s_q;
        if (q >= rp.num_tiles) break;   // uniform across the CTA
        // route_tile begins with a barrier, so every thread has read s_q before
        // thread 0 replaces it below
        route_tile<KT>(rp, q, epoch, reinterpret_cast<uint32_t *>(smem));
        if (tid == 0) s_q = (int)atomicAdd(&rp.hdr->ticket, 1u);
        __syncthreads();
    }
    // shared memory now changes hands from the routing step (generic writes) to
    // the mover's bulk copies (async proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if ((tid >> 5) < mp.pipes) move_body<MOVE_FUSED>(mp, smem, epoch);   // mp.wait_tiles is set by the launcher
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(&rp.hdr->done, 1u) == gridDim.x - 1) {
            atomicExch(&rp.hdr->ticket, 0u);
            atomicExch(&rp.hdr->move_next, 0u);
            atomicExch(&rp.hdr->routers, 0u);
            atomicExch(&rp.hdr->done, 0u);
            atomicExch(&rp.hdr->epoch, (epoch + 1u) & 0x3FFFFFFFu);
        }
    }
}

template <int KT>
static cudaError_t launch_dispatch_fused_kt(const RouteParams &rp, const MoveParams &mp, int grid,
                                            size_t smem, cudaStream_t st) {
    cudaError_t e = ensure_dyn_smem((const void *)dispatch_fused_kernel<KT>, smem);
    if (e != cudaSuccess) return e;
    dispatch_fused_kernel<KT><<<grid, kRouteThreads, smem, st>>>(rp, mp);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_fused(const RouteParams &rp, const MoveParams &mp, int grid,
                                  size_t move_smem, cudaStream_t st) {
    size_t smem = route_smem_bytes(rp.n_ctr, rp.K);
    if (move_smem > smem) smem = move_smem;
    switch (route_kt(rp.K)) {
        case 1: return launch_dispatch_fused_kt<1>(rp, mp, grid, smem, st);
        case 2: return launch_dispatch_fused_kt<2>(rp, mp, grid, smem, st);
        case 4: return launch_dispatch_fused_kt<4>(rp, mp, grid, smem, st);
        case 8: return launch_dispatch_fused_kt<8>(rp, mp, grid, smem, st);
        case 16: return launch_dispatch_fused_kt<16>(rp, mp, grid, smem, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_move(int mode, const MoveParams &p, int grid, int block, size_t smem, bool pdl,
                        cudaStream_t st) {
    const void *fn = nullptr;
    switch (mode) {
        case MOVE_FUSED: fn = (const void *)move_kernel<MOVE_FUSED>; break;
        case MOVE_PACK: fn = (const void *)move_kernel<MOVE_PACK>; break;
        case MOVE_EXCHANGE: fn = (const void *)move_kernel<MOVE_EXCHANGE>; break;
        case MOVE_DELIVER: fn = (const void *)move_kernel<MOVE_DELIVER>; break;
        default: return cudaErrorInvalidValue;
    }
    cudaError_t se = ensure_dyn_smem(fn, smem);
    if (se != cudaSuccess) return se;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<MoveParams *>(&p)};
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace ep
