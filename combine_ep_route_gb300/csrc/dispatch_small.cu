// dispatch_small.cu -- the fused dispatch for small batches (decode sizes):
// routing and row movement in one launch, with no communication between CTAs.
//
// It computes exactly what the routing tiles and the row mover compute
// (route_tile.cuh, move.cu): the slot of every (destination, token) in token
// order, the row of every pair inside its expert's batch in (source rank,
// slot) order, the received-slot metadata, the counts, and the delivered rows.
// Both numberings are exclusive prefix counts over tokens in (rank, token)
// order. On a small batch the ids of all tokens are a few tens of KiB, so
// every CTA counts the prefix of its own first token directly from the ids of
// all earlier tokens (read through L2) instead of waiting on a chain of
// look-back flags published by other CTAs. A CTA owns at most 32 consecutive
// token slots:
//   0. the threads load the token counts, the own tokens' ids and weights and
//      the first batch of earlier tokens' ids at launch; after the first barrier
//      thread 0 starts bulk copies of the CTA's token rows (and extra payloads)
//      into shared memory, which arrive while the prefix is counted;
//   1. every thread counts, over a strided share of the earlier tokens, the
//      kept pairs of each expert and -- for earlier tokens of the first token's
//      rank -- the destinations each reaches (warp-private counters in shared
//      memory, summed afterwards);
//   2. one thread per own (token, k) pair validates the id (staged in shared
//      memory at launch) and sets the token's lane bit in per-expert and
//      per-destination masks (a token reaching a rank twice sets one bit: the
//      (destination, token) deduplication);
//   3. every own (token, k) pair derives its row and slot from the prefix and
//      the masks twice, in two warps' threads: one stores the row to its expert's
//      batch with a bulk copy from shared memory, the other writes the pair
//      outputs and, for the first pair of a token on a destination, that
//      destination's received-slot row;
//   4. the CTA holding a rank's last token slot writes that rank's send counts,
//      and the one holding the very last slot writes expert_num_tokens.
// The only wait is the bounded one on the row copies' mbarrier.
#include "route_tile.cuh"

namespace ep {

namespace {

// A CTA has NT threads (256, 512 or 1024: more threads share the prefix count);
// each loads the ids of 1024 / NT earlier tokens per round.
constexpr int kSmallMinThreads = 256;
constexpr int kSmallRoundTokens = 1024;   // earlier tokens whose ids a CTA loads per round
static_assert(kSmallMinThreads >= EP_MAX_W, "one thread per rank loads the token counts");
static_assert(kSmallMaxTokens <= 32, "an own token is one bit of a 32-bit lane mask");

// Top-k ids of flat token g into ek (-1 past K); g < 0 gives all -1.
template <int KT>
__device__ __forceinline__ void load_ids(const RouteParams &p, int g, int (&ek)[KT]) {
    if (g >= 0 && KT % 4 == 0 && p.K == KT && p.vec_ids) {
        const int4 *pi = reinterpret_cast<const int4 *>(p.ids + (size_t)g * KT);
#pragma unroll
        for (int v = 0; v < KT / 4; ++v) {
            const int4 a = __ldg(pi + v);
            ek[4 * v] = a.x, ek[4 * v + 1] = a.y, ek[4 * v + 2] = a.z, ek[4 * v + 3] = a.w;
        }
        return;
    }
#pragma unroll
    for (int k = 0; k < KT; ++k) ek[k] = (g >= 0 && k < p.K) ? __ldg(p.ids + (size_t)g * p.K + k) : -1;
}

// Bit k set for each pair of the row that takes part: 0 <= id < E and not a
// repeat of an earlier kept id of the same row (the routing rule).
template <int KT>
__device__ __forceinline__ uint32_t kept_pairs(const int (&ek)[KT], int K, int E) {
    uint32_t keep = 0;
#pragma unroll
    for (int k = 0; k < KT; ++k) {
        const int e = ek[k];
        bool ok = k < K && e >= 0 && e < E;
#pragma unroll
        for (int k2 = 0; k2 < KT; ++k2)
            if (k2 < k && ((keep >> k2) & 1u) && ek[k2] == e) ok = false;
        if (ok) keep |= 1u << k;
    }
    return keep;
}

}  // namespace

// Shared memory: the CTA's rows, an mbarrier, warp-private counters
// [warps][W+E], the prefix [W+E], the own-token masks [W+E], the own pairs
// [32][KT] (packed destination and expert) with their weights, the clamped
// token counts [W], and the own tokens' ids as read [32][KT].
size_t small_smem_bytes(int n_per, uint32_t stage_bytes, int n_ctr, int top_k, int W, int threads) {
    const size_t rows = ((size_t)n_per * stage_bytes + 127) / 128 * 128;
    return rows + 16 + (size_t)(threads / 32 + 2) * n_ctr * 4 +
           (size_t)kSmallMaxTokens * route_kt(top_k) * 12 + (size_t)W * 4;
}

template <int KT, int NT>
__global__ void __launch_bounds__(NT) dispatch_small_kernel(const SmallParams sp) {
    constexpr int kSmallThreads = NT;
    constexpr int kSmallWarps = NT / 32;
    constexpr int kSmallIdBatch = kSmallRoundTokens / NT;
    extern __shared__ __align__(128) uint8_t smem[];
    const RouteParams &p = sp.rp;
    const MoveParams &m = sp.mp;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int W = p.W, E = p.E, K = p.K, Tm = p.Tm, e_local = p.e_local, n_ctr = p.n_ctr;
    const int n_slots = W * Tm;
    const int g0 = blockIdx.x * sp.n_per;
    const int g1 = min(g0 + sp.n_per, n_slots);
    const int n_own = g1 - g0;   // 1..32: the grid is ceil(n_slots / n_per)
    const uint32_t sb = sp.stage_bytes;

    uint8_t *rows = smem;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + ((size_t)sp.n_per * sb + 127) / 128 * 128);
    int32_t *cnt = reinterpret_cast<int32_t *>(bar + 2);   // [warps][n_ctr]
    int32_t *excl = cnt + kSmallWarps * n_ctr;             // [n_ctr]
    uint32_t *bits = reinterpret_cast<uint32_t *>(excl + n_ctr);   // [n_ctr]
    int32_t *sid = reinterpret_cast<int32_t *>(bits + n_ctr);      // [32][KT]
    float *sw = reinterpret_cast<float *>(sid + kSmallMaxTokens * KT);   // [32][KT]
    int32_t *sT = reinterpret_cast<int32_t *>(sw + kSmallMaxTokens * KT);   // [W]
    int32_t *sraw = sT + W;                                                  // [32][KT]

    // a combine launched with programmatic dependent launch may start its
    // prologue now; it waits for this grid's completion before reading anything
    pdl_launch_dependents();

    // 0. every small global read starts at once: the token counts, the own
    // tokens' ids and weights, and the first batch of earlier tokens' ids; the
    // CTA's rows follow right after the first barrier (below)
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    int T_in = Tm;
    if (tid < W && p.num_tokens) T_in = __ldg(p.num_tokens + tid);
    if (tid < n_own) {   // the own token's ids and weights, as read
        int own_ids[KT];
        load_ids<KT>(p, g0 + tid, own_ids);
#pragma unroll
        for (int k = 0; k < KT; ++k) {
            sraw[tid * KT + k] = own_ids[k];
            sw[tid * KT + k] = k < K ? __ldg(p.weights + (size_t)(g0 + tid) * K + k) : 0.f;
        }
    }
    int ek[kSmallIdBatch][KT];
#pragma unroll
    for (int b = 0; b < kSmallIdBatch; ++b) {
        const int gp = b * kSmallThreads + tid;
        load_ids<KT>(p, gp < g0 ? gp : -1, ek[b]);
    }
    for (int i = tid; i < kSmallWarps * n_ctr; i += kSmallThreads) cnt[i] = 0;
    for (int i = tid; i < n_ctr; i += kSmallThreads) bits[i] = 0u;
    if (tid < W) {
        int T = T_in;
        if (T < 0 || T > Tm) {
            // reported once, by the CTA holding the rank's first slot
            if (tid * Tm >= g0 && tid * Tm < g1) raise_error(p.hdr, EP_ERR_CAPACITY);
            T = T < 0 ? 0 : Tm;
        }
        sT[tid] = T;
    }
    __syncthreads();
    // The rows (bulk copies into shared memory) are needed only once the prefix
    // is counted; issued at launch they delayed the ids' round trip that the
    // count waits on (decode step 21.3 -> 20.7 us on GB300 when issued here).
    if (tid == 0) {
        mbar_arrive_expect_tx(bar, (uint32_t)n_own * m.row_bytes);
        for (int i = 0; i < n_own; ++i)
            for (int sg = 0; sg < m.n_seg; ++sg)
                bulk_g2s(rows + (size_t)i * sb + m.seg_off[sg],
                         m.src_seg[sg] + (size_t)(g0 + i) * m.seg_bytes[sg], m.seg_bytes[sg], bar);
    }

    // 1. the prefix of the first own token, counted from the earlier tokens' ids
    const int s0 = (int)fastdiv((uint32_t)g0, sp.div_tm);
    int32_t *mycnt = cnt + warp * n_ctr;
    for (int base = 0; base < g0; base += kSmallThreads * kSmallIdBatch) {
        if (base > 0) {
#pragma unroll
            for (int b = 0; b < kSmallIdBatch; ++b) {
                const int gp = base + b * kSmallThreads + tid;
                load_ids<KT>(p, gp < g0 ? gp : -1, ek[b]);
            }
        }
#pragma unroll
        for (int b = 0; b < kSmallIdBatch; ++b) {
            const int gp = base + b * kSmallThreads + tid;
            if (gp >= g0) continue;
            const int sq = (int)fastdiv((uint32_t)gp, sp.div_tm);
            if (gp - sq * Tm >= sT[sq]) continue;
            const uint32_t keep = kept_pairs<KT>(ek[b], K, E);
            uint64_t dm = 0;
#pragma unroll
            for (int k = 0; k < KT; ++k) {
                if (!((keep >> k) & 1u)) continue;
                const int e = ek[b][k];
                atomicAdd(&mycnt[W + e], 1);
                if (sq == s0) {
                    const int d = (int)fastdiv((uint32_t)e, sp.div_el);
                    if (!((dm >> d) & 1ull)) {
                        dm |= 1ull << d;
                        atomicAdd(&mycnt[d], 1);
                    }
                }
            }
        }
    }

    // 2. one thread per own (token, k) pair: validate, and set the token's lane
    // bit for its expert and destination. A valid id repeated at a later k of the
    // same token is the duplicate (the first occurrence of a valid id is always
    // kept), and a token that reaches a rank twice sets one bit: the
    // (destination, token) deduplication.
    for (int pi = tid; pi < n_own * KT; pi += kSmallThreads) {
        const int tl = pi / KT, k = pi - (pi / KT) * KT;
        const int g = g0 + tl;
        const int s = (int)fastdiv((uint32_t)g, sp.div_tm);
        const int32_t *raw = sraw + tl * KT;
        const int e = (k < K && g - s * Tm < sT[s]) ? raw[k] : -1;
        bool ok = e >= 0;
        if (ok && e >= E) {
            raise_error(p.hdr, EP_ERR_EXPERT_ID);
            ok = false;
        }
        if (ok) {
            bool dup = false;
#pragma unroll
            for (int k2 = 0; k2 < KT; ++k2) dup |= k2 < k && raw[k2] == e;
            if (dup) {
                raise_error(p.hdr, EP_ERR_DUPLICATE);
                ok = false;
            }
        }
        int packed = -1;
        if (ok) {
            const int d = (int)fastdiv((uint32_t)e, sp.div_el);
            atomicOr(&bits[d], 1u << tl);
            atomicOr(&bits[W + e], 1u << tl);
            packed = (d << 16) | e;
        }
        sid[pi] = packed;
    }
    __syncthreads();
    for (int c = tid; c < n_ctr; c += kSmallThreads) {
        int v = 0;
#pragma unroll
        for (int w2 = 0; w2 < kSmallWarps; ++w2) v += cnt[w2 * n_ctr + c];
        excl[c] = v;
    }
    __syncthreads();

    // 3. the own (token, k) pairs: row copies and metadata
    auto rank_mask = [&](int s) -> uint32_t {   // own tokens of rank s
        const int lo = max(s * Tm - g0, 0), hi = min((s + 1) * Tm - g0, n_own);
        if (hi <= lo) return 0u;
        const uint32_t upto = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
        return upto & ~((1u << lo) - 1u);
    };
    auto locate = [&](int tl, int pk, int &slot, int &row) -> bool {
        if (pk < 0) return false;
        const int e = pk & 0xFFFF, d = pk >> 16;
        const int s = (int)fastdiv((uint32_t)(g0 + tl), sp.div_tm);
        const uint32_t lt = (1u << tl) - 1u;
        slot = (s == s0 ? excl[d] : 0) + __popc(bits[d] & lt & rank_mask(s));
        row = excl[W + e] + __popc(bits[W + e] & lt);
        return slot >= 0 && slot < sT[s] && row >= 0 && row < p.Ecap;
    };
    auto first_on_dest = [&](const int32_t *te, int k, int d) -> bool {
        bool first = true;
#pragma unroll
        for (int k2 = 0; k2 < KT; ++k2)
            if (k2 < k && te[k2] >= 0 && (te[k2] >> 16) == d) first = false;
        return first;
    };
    // Each pair has two jobs, held by threads of different warps: the first n_pad
    // threads store the rows (bulk copies from shared memory), the next n_pad write
    // the pair outputs and received-slot rows. A warp's bulk-copy instruction
    // completes only once the copy engine has taken all its lanes' copies (~3.5 us
    // for 32 rows of 4 KiB), so metadata stores issued by the same threads after it
    // would finish only then.
    const int n_pairs = n_own * KT;
    const int n_pad = (n_pairs + 31) & ~31;
    bool waited = false, loaded = false, stored = false;
    for (int wi = tid; wi < 2 * n_pad; wi += kSmallThreads) {
        const bool meta = wi >= n_pad;
        const int pi = meta ? wi - n_pad : wi;
        if (pi >= n_pairs) continue;
        const int tl = pi / KT, k = pi - (pi / KT) * KT;
        if (k >= K) continue;
        const int g = g0 + tl;
        const int s = (int)fastdiv((uint32_t)g, sp.div_tm);
        const int32_t *te = sid + tl * KT;
        const int pk = te[k];
        int slot = 0, row = 0;
        const bool found = locate(tl, pk, slot, row);
        if (!meta) {
            // the row, from shared memory to the pair's row of its expert
            if (!found) continue;
            const int prow = (pk & 0xFFFF) * p.Ecap + row;
            if (!waited) {
                loaded = mbar_wait_bounded(bar, 0u, p.wait_limit_ns, p.hdr);
                waited = true;
            }
            if (loaded) {
                const uint8_t *stg = rows + (size_t)tl * sb;
                for (int sg = 0; sg < m.n_seg; ++sg)
                    bulk_s2g(m.dst_seg[sg] + (size_t)prow * m.seg_bytes[sg], stg + m.seg_off[sg],
                             m.seg_bytes[sg]);
                stored = true;
            }
            continue;
        }
        int32_t prow = -1, psend = -1;
        float pw = 0.f;
        if (found) {
            const int e = pk & 0xFFFF, d = pk >> 16;
            prow = e * p.Ecap + row;
            pw = p.unit_weights ? 1.0f : sw[tl * KT + k];
            const bool first = first_on_dest(te, k, d);
            if (first) psend = (s * W + d) * Tm + slot;
            if (first) {
                // the received-slot row on d: the token's pairs on d in top-k order
                const uint32_t lt = (1u << tl) - 1u;
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
                        const int r2 = excl[W + e2] + __popc(bits[W + e2] & lt);
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
                const size_t rb = ((size_t)(d * W + s) * Tm + slot) * p.S;
                if (KT >= 4 && p.vec_recv) {
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
        } else if (pk >= 0) {
            raise_error(p.hdr, EP_ERR_STATE);   // a prefix out of range; never expected
        }
        p.pair_row[(size_t)g * K + k] = prow;
        p.pair_w[(size_t)g * K + k] = pw;
        p.pair_send[(size_t)g * K + k] = psend;
    }
    if (stored) bulk_commit();

    // 4. counts: a rank's send counts from the CTA holding its last slot, the
    // experts' row counts from the CTA holding the very last slot
    const int s_last = (int)fastdiv((uint32_t)(g1 - 1), sp.div_tm);
    for (int s = s0; s <= s_last; ++s) {
        if ((s + 1) * Tm - 1 >= g1) continue;
        const uint32_t rm = rank_mask(s);
        for (int d = tid; d < W; d += kSmallThreads)
            p.send_cnt[s * W + d] = min(max((s == s0 ? excl[d] : 0) + __popc(bits[d] & rm), 0), sT[s]);
    }
    if (g1 == n_slots) {
        const uint32_t all = n_own >= 32 ? 0xffffffffu : ((1u << n_own) - 1u);
        for (int e = tid; e < E; e += kSmallThreads)
            p.expert_num_tokens[e] = min(max(excl[W + e] + __popc(bits[W + e] & all), 0), p.Ecap);
    }

    // the row copies must be done before the CTA's shared memory goes away: the
    // stores this thread issued, and the loads into shared memory, which thread 0
    // waits for (bounded) unless it has seen them complete -- also after a wait
    // that ran out, so a CTA never exits with its loads still in flight unless a
    // second full wait runs out as well
    if (stored) bulk_wait_all();
    if (tid == 0 && !loaded) mbar_wait_bounded(bar, 0u, p.wait_limit_ns, p.hdr);
}

template <int KT, int NT>
static const void *small_kernel() {
    if constexpr (KT == 16 && NT > 512) return nullptr;   // registers: see small_threads
    else return (const void *)dispatch_small_kernel<KT, NT>;
}

template <int NT>
static const void *small_fn(int top_k) {
    switch (route_kt(top_k)) {
        case 1: return small_kernel<1, NT>();
        case 2: return small_kernel<2, NT>();
        case 4: return small_kernel<4, NT>();
        case 8: return small_kernel<8, NT>();
        case 16: return small_kernel<16, NT>();
        default: return nullptr;
    }
}

// Threads per CTA of the small-batch dispatch: as many as the registers of one
// CTA per SM allow (the kernel for top_k 16 needs more registers per thread).
int small_threads(int top_k) { return route_kt(top_k) <= 8 ? 1024 : 512; }

cudaError_t launch_dispatch_small(const SmallParams &sp, int grid, int threads, size_t smem,
                                  cudaStream_t st) {
    const void *fn = threads == 1024 ? small_fn<1024>(sp.rp.K)
                   : threads == 512  ? small_fn<512>(sp.rp.K)
                   : threads == 256  ? small_fn<256>(sp.rp.K)
                                     : nullptr;
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = ensure_dyn_smem(fn, smem);
    if (e != cudaSuccess) return e;
    void *args[] = {const_cast<SmallParams *>(&sp)};
    e = cudaLaunchKernel(fn, dim3(grid), dim3(threads), args, smem, st);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace ep
