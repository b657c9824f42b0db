"""A second, independent CPU formulation of the dispatch metadata, by stable sorting.

TEST INFRASTRUCTURE ONLY. Its one purpose is to pin the counter-loop oracle
(``ep_oracle.c``): the two are written in different ways and must agree bit for
bit on every input.

It restates the sort-based description of vLLM
``AllToAllBatchedPrepareAndFinalize.prepare`` (page
fused_moe/prepare_finalize/alltoall_batched): order the kept (token, expert)
pairs of a rank by (destination rank, token), take the first pair of each
(destination, token) run as that token's slot on the destination, number the
slots of a destination from zero, and place the pairs of a run in consecutive
columns. On the receiving side the valid (source, slot, column) entries are
walked in order and each local expert's rows are numbered in that order.

Here the ordering is an explicit stable ``np.lexsort`` (so the columns of a
run follow top-k order, the reading the counter oracle also takes), the runs
come from ``np.unique`` and the per-expert row numbers from a stable sort by
expert, in place of the counters of the loop formulation.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

ERR_EXPERT_ID = 1
ERR_DUPLICATE = 2
ERR_CAPACITY = 4


def dispatch_meta_sorted(W: int, E: int, K: int, Tm: int, topk_ids: np.ndarray,
                         topk_weights: np.ndarray,
                         num_tokens: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    e_local = E // W
    S = min(K, e_local)
    Ecap = Tm * W
    ids = np.asarray(topk_ids, dtype=np.int64).reshape(W, Tm, K)
    wts = np.asarray(topk_weights, dtype=np.float32).reshape(W, Tm, K)
    nt = np.full(W, Tm) if num_tokens is None else np.asarray(num_tokens).reshape(W)
    err = 0
    send_cnt = np.zeros((W, W), np.int32)
    send_tok = np.full((W, W, Tm), -1, np.int32)
    send_eloc = np.full((W, W, Tm, S), -1, np.int32)
    send_w = np.zeros((W, W, Tm, S), np.float32)
    send_k = np.full((W, W, Tm, S), -1, np.int32)

    for s in range(W):
        T = int(nt[s])
        if T < 0 or T > Tm:
            err |= ERR_CAPACITY
            T = 0 if T < 0 else Tm
        if T == 0:
            continue
        e = ids[s, :T].reshape(-1)
        t = np.repeat(np.arange(T), K)
        k = np.tile(np.arange(K), T)
        w = wts[s, :T].reshape(-1)
        keep = e >= 0
        bad = keep & (e >= E)
        if bad.any():
            err |= ERR_EXPERT_ID
        keep &= ~bad
        # a repeated id in a row: keep its first (lowest k) occurrence only
        o = np.lexsort((k, e, t))            # by token, then id, then k
        same = np.zeros(len(o), bool)
        same[1:] = (t[o][1:] == t[o][:-1]) & (e[o][1:] == e[o][:-1]) & keep[o][1:] & keep[o][:-1]
        dup = np.zeros(len(o), bool)
        dup[o] = same
        if (dup & keep).any():
            err |= ERR_DUPLICATE
        keep &= ~dup
        e, t, k, w = e[keep], t[keep], k[keep], w[keep]
        if len(e) == 0:
            continue
        d = e // e_local
        o = np.lexsort((k, t, d))            # by destination, then token, then k (stable)
        d, t, k, e, w = d[o], t[o], k[o], e[o], w[o]
        runs, first, run_of = np.unique(d * (Tm + 1) + t, return_index=True, return_inverse=True)
        run_d = d[first]
        run_t = t[first]
        cnt = np.bincount(run_d, minlength=W)
        start = np.concatenate(([0], np.cumsum(cnt)))
        run_slot = np.arange(len(runs)) - start[run_d]
        send_cnt[s] = cnt
        send_tok[s, run_d, run_slot] = run_t
        col = np.arange(len(e)) - first[run_of]
        slot = run_slot[run_of]
        send_eloc[s, d, slot, col] = e - d * e_local
        send_w[s, d, slot, col] = w
        send_k[s, d, slot, col] = k

    recv_cnt = np.ascontiguousarray(send_cnt.T)
    recv_eloc = np.ascontiguousarray(send_eloc.transpose(1, 0, 2, 3))
    recv_w = np.ascontiguousarray(send_w.transpose(1, 0, 2, 3))

    ent = np.zeros((W, e_local), np.int32)
    row_src = np.full((E, Ecap), -1, np.int32)
    row_col = np.full((E, Ecap), -1, np.int32)
    slot_ar = np.arange(Tm)
    for dd in range(W):
        valid = (slot_ar[None, :] < recv_cnt[dd][:, None])[:, :, None] & (recv_eloc[dd] >= 0)
        vs, vq, vc = np.nonzero(valid)       # (source, slot, column) in order
        j = recv_eloc[dd][vs, vq, vc].astype(np.int64)
        oj = np.argsort(j, kind="stable")
        jj = j[oj]
        grp_start = np.searchsorted(jj, jj, side="left")
        row = np.arange(len(jj)) - grp_start
        if len(row) and row.max() >= Ecap:
            err |= ERR_CAPACITY
        ent[dd] = np.bincount(j, minlength=e_local)
        flat = (dd * e_local + jj) * Ecap + row
        row_src.reshape(-1)[flat] = vs[oj] * Tm + vq[oj]
        row_col.reshape(-1)[flat] = vc[oj]

    # token side: which row holds each (s, t, k)
    pair_row = np.full((W, Tm, K), -1, np.int32)
    fe, frow = np.nonzero(row_src >= 0)
    src = row_src[fe, frow]
    ss, qq, cc = src // Tm, src % Tm, row_col[fe, frow]
    dd = fe // e_local
    tt = send_tok[ss, dd, qq]
    kk = send_k[ss, dd, qq, cc]
    pair_row[ss, tt, kk] = fe * Ecap + frow
    return dict(send_cnt=send_cnt, send_tok=send_tok, send_eloc=send_eloc, send_w=send_w,
                send_k=send_k, recv_cnt=recv_cnt, recv_eloc=recv_eloc, recv_w=recv_w,
                expert_num_tokens=ent, row_src=row_src, row_col=row_col, pair_row=pair_row,
                err=np.int64(err))
