"""Pins of the CPU oracle against things other than itself.

* a hand-derived worked example (tests/golden/worked_example.json);
* an independent stable-sort formulation (oracle/sort_oracle.py), bit for bit,
  exhaustively on tiny inputs and on random and full-size inputs;
* the invariants the routed all-to-all dispatch must satisfy (vLLM
  AllToAllBatchedPrepareAndFinalize.prepare: one slot per (dest, token) in
  token order, k-th expert in column k, per-expert rows in (source, slot)
  order, capacities);
* special cases that reduce to a library routine (W = 1 is a stable counting
  sort of the pairs by expert id) or to closed forms (one-hot weights, identity
  experts with weights summing to one, exact power-of-two scaling);
* the combine fold against an fp64 evaluation of its plain definition, within
  the standard error bound of a K-term fp32 sum.
"""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import ref, sort_oracle
from combine_ep_route_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")
META_KEYS = ("send_cnt", "send_tok", "send_eloc", "send_w", "send_k", "recv_cnt", "recv_eloc",
             "recv_w", "expert_num_tokens", "row_src", "row_col", "pair_row")


def _meta(W, E, K, T, ids, w=None, nt=None):
    if w is None:
        w = np.ones(np.shape(ids), np.float32)
    return ref.dispatch_meta(W, E, K, T, np.asarray(ids, np.int32), np.asarray(w, np.float32), nt)


def _agree(W, E, K, T, ids, w, nt=None):
    m = ref.dispatch_meta(W, E, K, T, ids, w, nt)
    so = sort_oracle.dispatch_meta_sorted(W, E, K, T, ids, w, nt)
    for k in META_KEYS:
        a, b = getattr(m, k), so[k]
        assert a.shape == b.shape and np.array_equal(a, b), (k, ids.tolist(), a, b)
    assert m.err == int(so["err"])
    return m


# ---------------------------------------------------------------- capacities

@pytest.mark.parametrize("W,E,K,T,expect", [
    (8, 64, 8, 128, (128, 8, 1024)),
    (4, 8, 8, 16, (16, 2, 64)),     # K > e_local: slots per token clamp to e_local
    (1, 4, 2, 5, (5, 2, 5)),
    (32, 256, 8, 256, (256, 8, 8192)),
])
def test_capacities(W, E, K, T, expect):
    assert ref.capacities(W, E, K, T) == expect


# ----------------------------------------------------------- worked example

def test_worked_example_dispatch():
    g = json.load(open(GOLDEN))
    W, E, K, T = g["W"], g["E"], g["K"], g["Tm"]
    assert ref.capacities(W, E, K, T) == tuple(g["capacities"])
    m = _meta(W, E, K, T, g["topk_ids"])
    assert m.err == 0
    assert m.send_cnt.tolist() == g["send_cnt"]
    for key, toks in g["send_tok"].items():
        s, d = map(int, key.split("->"))
        assert m.send_tok[s, d, :len(toks)].tolist() == toks
        assert (m.send_tok[s, d, len(toks):] == -1).all()
    for key, cols in g["send_eloc"].items():
        s, d = map(int, key.split("->"))
        assert m.send_eloc[s, d, :len(cols)].tolist() == cols
    assert m.expert_num_tokens.tolist() == g["expert_num_tokens"]
    rt = m.row_token()
    e_local = E // W
    for key, srcs in g["expert_rows_src_token"].items():
        d, j = map(int, key.split(","))
        got = rt[d * e_local + j, :len(srcs)]
        assert got.tolist() == [s * T + t for s, t in srcs]
        assert (rt[d * e_local + j, len(srcs):] == -1).all()
    assert m.n_rows == 8


def test_worked_example_payload_and_combine():
    g = json.load(open(GOLDEN))
    W, E, K, T, h = g["W"], g["E"], g["K"], g["Tm"], g["h"]
    a1 = wl.f32_to_bf16_bits(np.array(g["a1"], np.float32))
    w = np.array(g["topk_weights"], np.float32)
    m = _meta(W, E, K, T, g["topk_ids"], w)
    rows = ref.dispatch_rows(m, a1)
    # expert (d, j) scales its input by (global id + 1)
    scale = np.concatenate([np.full(int(m.expert_num_tokens.reshape(-1)[e]), e + 1.0)
                            for e in range(E)]).astype(np.float32)
    x = wl.bf16_bits_to_f32(rows.view(np.uint16).reshape(-1, h)) * scale[:, None]
    xb = wl.f32_to_bf16_bits(x)
    expect = np.array(g["combine_out"], np.float32).reshape(W * T, h)
    out32 = ref.combine(m, w, xb, out_f32=True)
    assert np.array_equal(out32, expect)
    outb = ref.combine(m, w, xb, out_f32=False)
    assert np.array_equal(wl.bf16_bits_to_f32(outb), expect)


# ------------------------------------------------- two formulations, exhaustive

def _token_options(E, K):
    """Every top-k row over E experts with distinct ids, allowing -1 padding entries."""
    opts = []
    for row in itertools.product(range(-1, E), repeat=K):
        v = [e for e in row if e >= 0]
        if len(set(v)) == len(v):
            opts.append(row)
    return opts


def test_exhaustive_tiny_w2_e4_k2_t3():
    W, E, K, T = 2, 4, 2, 3
    opts = _token_options(E, K)
    assert len(opts) == 21
    others = [((3, 0), (1, 2), (-1, -1)), ((0, 1), (2, 3), (1, -1)), ((-1, -1),) * 3]
    w = np.linspace(0.1, 0.9, W * T * K, dtype=np.float32).reshape(W, T, K)
    n = 0
    for i, r0 in enumerate(itertools.product(opts, repeat=T)):
        ids = np.array([r0, others[i % len(others)]], np.int32)
        for swap in (False, True):
            x = ids[::-1].copy() if swap else ids
            m = _agree(W, E, K, T, x, w)
            assert m.err == 0
            n += 1
    assert n == 2 * 21 ** 3


def test_random_tiny_cases_agree_including_errors():
    rng = np.random.default_rng(7)
    for case in range(10000):
        W = int(rng.integers(1, 5))
        e_local = int(rng.integers(1, 4))
        E = W * e_local
        K = int(rng.integers(1, min(E, 4) + 1))
        T = int(rng.integers(1, 6))
        ids = rng.integers(-2, E + (1 if case % 5 == 0 else 0), size=(W, T, K)).astype(np.int32)
        if case % 7 == 0:
            ids[..., -1] = ids[..., 0]        # plant repeated ids
        w = rng.random((W, T, K), dtype=np.float32)
        nt = rng.integers(0, T + 1, size=W).astype(np.int32) if case % 3 == 0 else None
        _agree(W, E, K, T, ids, w, nt)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_named_workloads_agree(cfg):
    x = wl.make(cfg)
    s = x.spec
    m = _agree(s.W, s.E, s.K, s.T, x.topk_ids, x.topk_weights, x.num_tokens)
    assert m.err == 0
    _check_invariants(m, x.topk_ids, x.num_tokens)


# ------------------------------------------------------------------ invariants

def _check_invariants(m, ids, nt):
    W, E, K, T, S, Ecap = m.W, m.E, m.K, m.Tm, m.S, m.Ecap
    e_local = E // W
    ids = np.asarray(ids).reshape(W, T, K)
    for s in range(W):
        dt = set()
        for t in range(int(nt[s])):
            for e in ids[s, t]:
                if 0 <= e < E:
                    dt.add((int(e) // e_local, t))
        # per-dest counts sum to the deduplicated (dest, token) pairs
        assert int(m.send_cnt[s].sum()) == len(dt)
        for d in range(W):
            c = int(m.send_cnt[s, d])
            toks = m.send_tok[s, d, :c]
            # slots: each token at most once per dest, in increasing token order
            assert np.all(np.diff(toks) > 0)
            assert sorted(t for (dd, t) in dt if dd == d) == toks.tolist()
            assert (m.send_tok[s, d, c:] == -1).all()
            for q, t in enumerate(toks):
                # column c holds the c-th of the token's experts on d, in top-k order
                want = [int(e) - d * e_local for e in ids[s, t] if 0 <= e < E and e // e_local == d]
                got = m.send_eloc[s, d, q]
                assert got[:len(want)].tolist() == want
                assert (got[len(want):] == -1).all()
                ks = m.send_k[s, d, q, :len(want)]
                assert np.all(np.diff(ks) > 0)
        # padding tokens (all ids negative) are sent nowhere
        pad = [t for t in range(T) if (ids[s, t] < 0).all()]
        assert not np.isin(m.send_tok[s], pad).any()
    # capacity bound and per-dest pair count
    assert (m.expert_num_tokens <= Ecap).all()
    for d in range(W):
        n_pairs = sum(1 for s in range(W) for t in range(int(nt[s])) for e in ids[s, t]
                      if 0 <= e < E and e // e_local == d)
        assert int(m.expert_num_tokens[d].sum()) == n_pairs
    # rows of each expert sorted by (source rank, slot)
    for e in range(E):
        n = int(m.expert_num_tokens.reshape(-1)[e])
        src = m.row_src[e, :n]
        assert np.all(np.diff(src) > 0)
        assert (m.row_src[e, n:] == -1).all()
    # every routed pair has exactly one row and the row holds its token
    rt = m.row_token()
    pr = m.pair_row.reshape(-1)
    kept = pr >= 0
    assert len(np.unique(pr[kept])) == kept.sum() == m.n_rows
    g = np.repeat(np.arange(W * T), K)[kept]
    assert np.array_equal(rt.reshape(-1)[pr[kept]], g)


def test_invariants_random_medium():
    rng = np.random.default_rng(11)
    for _ in range(20):
        W = int(rng.integers(1, 7))
        e_local = int(rng.integers(1, 6))
        E = W * e_local
        K = int(rng.integers(1, min(E, 6) + 1))
        T = int(rng.integers(1, 40))
        ids = np.stack([rng.permutation(E)[:K] for _ in range(W * T)]).reshape(W, T, K)
        ids[rng.random((W, T)) < 0.2] = -1
        ids = ids.astype(np.int32)
        nt = rng.integers(0, T + 1, size=W).astype(np.int32)
        m = _meta(W, E, K, T, ids, None, nt)
        assert m.err == 0
        _check_invariants(m, ids, nt)


# --------------------------------------------------------------- special cases

def test_w1_is_a_stable_counting_sort_by_expert():
    rng = np.random.default_rng(3)
    E, K, T = 6, 3, 50
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)[None]
    m = _meta(1, E, K, T, ids)
    flat = ids.reshape(-1)
    order = np.argsort(flat, kind="stable")            # pairs by expert, token order kept
    tok = (np.arange(T * K) // K)[order]
    exp_sorted = flat[order]
    rt = m.row_token()
    for e in range(E):
        assert rt[e, :int(m.expert_num_tokens[0, e])].tolist() == tok[exp_sorted == e].tolist()
    assert np.array_equal(m.expert_num_tokens[0], np.bincount(flat, minlength=E))


def test_errors_flagged_and_pairs_dropped():
    W, E, K, T = 2, 4, 3, 2
    ids = np.array([[[0, 9, -3], [1, 1, 2]], [[-1, -1, -1], [3, 0, -2]]], np.int32)
    m = _meta(W, E, K, T, ids)
    assert m.err & ref.ERR_EXPERT_ID and m.err & ref.ERR_DUPLICATE
    pr = m.pair_row
    assert pr[0, 0, 0] >= 0 and pr[0, 0, 1] == -1 and pr[0, 0, 2] == -1
    assert pr[0, 1, 0] >= 0 and pr[0, 1, 1] == -1 and pr[0, 1, 2] >= 0
    assert (pr[1, 0] == -1).all() and pr[1, 1, 2] == -1
    m2 = _meta(W, E, K, T, np.zeros((W, T, K), np.int32) - 1, None, np.array([3, 1], np.int32))
    assert m2.err & ref.ERR_CAPACITY


def test_payload_rows_are_the_source_tokens():
    x = wl.make(wl.spec(4, T=64))
    s = x.spec
    m = ref.dispatch_meta(s.W, s.E, s.K, s.T, x.topk_ids, x.topk_weights)
    src = np.concatenate([x.a1.view(np.uint8), x.extras[0]], axis=2)
    rows = ref.dispatch_rows(m, src)
    rt = m.row_token()
    flat_src = src.reshape(s.W * s.T, -1)
    for e in range(s.E):
        n = int(m.expert_num_tokens.reshape(-1)[e])
        o = int(m.row_off[e])
        assert np.array_equal(rows[o:o + n], flat_src[rt[e, :n]])


# ------------------------------------------------------------------ combine

def _rand_expert_rows(m, h, seed):
    rng = np.random.default_rng(seed)
    return wl.f32_to_bf16_bits(rng.standard_normal((m.n_rows, h), dtype=np.float32))


def _exact64(m, w, rows, h):
    """The plain definition of combine in fp64: sum_k w_k * row_k."""
    W, T, K = m.W, m.Tm, m.K
    x = wl.bf16_bits_to_f32(rows.reshape(m.n_rows, h)).astype(np.float64)
    out = np.zeros((W * T, h))
    absacc = np.zeros((W * T, h))
    pr = m.pair_row.reshape(W * T, K)
    wf = np.asarray(w, np.float64).reshape(W * T, K)
    for g in range(W * T):
        for k in range(K):
            f = pr[g, k]
            if f < 0:
                continue
            r = m.row_off[f // m.Ecap] + f % m.Ecap
            out[g] += wf[g, k] * x[r]
            absacc[g] += abs(wf[g, k] * x[r])
    return out, absacc


@pytest.mark.parametrize("cfg,T", [(1, None), (2, 32), (4, 16), (5, 8)])
def test_combine_within_fp32_sum_bound_of_exact(cfg, T):
    x = wl.make(wl.spec(cfg, T=T) if T else wl.spec(cfg))
    s = x.spec
    m = ref.dispatch_meta(s.W, s.E, s.K, s.T, x.topk_ids, x.topk_weights)
    rows = _rand_expert_rows(m, s.h, 5)
    out = ref.combine(m, x.topk_weights, rows, out_f32=True)
    exact, absacc = _exact64(m, x.topk_weights, rows, s.h)
    u = 2.0 ** -24
    gamma = 2 * s.K * u / (1 - 2 * s.K * u)     # K products and K sums, each rounded once
    assert np.all(np.abs(out - exact) <= gamma * absacc + 1e-45)
    # bf16 output is the fp32 fold rounded once
    outb = ref.combine(m, x.topk_weights, rows, out_f32=False)
    assert np.array_equal(outb, wl.f32_to_bf16_bits(out))
    # padding rows are zero
    pad = (x.topk_ids.reshape(-1, s.K) < 0).all(axis=1)
    assert (out[pad] == 0).all() and (outb[pad] == 0).all()


def test_combine_one_hot_weights_return_the_expert_row():
    x = wl.make(wl.spec(2, T=24))
    s = x.spec
    rng = np.random.default_rng(1)
    pick = rng.integers(0, s.K, size=(s.W, s.T))
    w = np.zeros_like(x.topk_weights)
    np.put_along_axis(w, pick[..., None], 1.0, axis=2)
    m = ref.dispatch_meta(s.W, s.E, s.K, s.T, x.topk_ids, w)
    rows = _rand_expert_rows(m, s.h, 2)
    outb = ref.combine(m, w, rows, out_f32=False)
    pr = m.pair_row.reshape(-1, s.K)
    for g in range(s.W * s.T):
        f = pr[g, pick.reshape(-1)[g]]
        if f < 0:
            assert (outb[g] == 0).all()
            continue
        r = m.row_off[f // m.Ecap] + f % m.Ecap
        assert np.array_equal(outb[g], rows[r])


@pytest.mark.parametrize("cfg", [1, 2])
def test_identity_experts_reproduce_a1(cfg):
    x = wl.make(cfg)
    s = x.spec
    m = ref.dispatch_meta(s.W, s.E, s.K, s.T, x.topk_ids, x.topk_weights)
    rows = ref.dispatch_rows(m, x.a1)
    outb = ref.combine(m, x.topk_weights, rows, out_f32=False).reshape(s.W, s.T, s.h)
    routed = (x.topk_ids >= 0).any(axis=2)
    assert np.array_equal(outb[routed], x.a1[routed])
    assert (outb[~routed] == 0).all()


def test_combine_scales_exactly_with_weights():
    x = wl.make(wl.spec(2, T=16))
    s = x.spec
    m = ref.dispatch_meta(s.W, s.E, s.K, s.T, x.topk_ids, x.topk_weights)
    rows = _rand_expert_rows(m, s.h, 9)
    o1 = ref.combine(m, x.topk_weights, rows, out_f32=True)
    o2 = ref.combine(m, 2 * x.topk_weights, rows, out_f32=True)
    assert np.array_equal(o2, 2 * o1)


def test_pagemode_two_stage_rounding_bounded():
    """The page's own finalize rounds per-destination partials to bf16 before the
    return exchange and sums them in the output type. Against the single-rounding
    fold it differs by a few bf16 roundings of the summed magnitudes: bounded
    element-wise by 2^-6 * sum_k |w_k x_k| and normwise by 1e-2. (Element-wise
    relative error is not bounded where outputs cancel towards zero.)"""
    for cfg, T in [(2, 32), (5, 8)]:
        x = wl.make(wl.spec(cfg, T=T))
        s = x.spec
        m = ref.dispatch_meta(s.W, s.E, s.K, s.T, x.topk_ids, x.topk_weights)
        rows = _rand_expert_rows(m, s.h, 4)
        _, absacc = _exact64(m, x.topk_weights, rows, s.h)
        for f32 in (False, True):
            ours = ref.combine(m, x.topk_weights, rows, out_f32=f32)
            page = ref.combine_pagemode(m, rows, out_f32=f32)
            if not f32:
                ours, page = wl.bf16_bits_to_f32(ours), wl.bf16_bits_to_f32(page)
            diff = np.abs(page.astype(np.float64) - ours)
            assert np.all(diff <= 2.0 ** -6 * absacc)
            assert np.linalg.norm(diff) <= 1e-2 * np.linalg.norm(ours)
    # one destination per token and one expert there: the two forms agree exactly
    x = wl.make(wl.spec(1))
    s = x.spec
    ids = x.topk_ids.copy()
    ids[..., 1:] = -1
    m = ref.dispatch_meta(s.W, s.E, s.K, s.T, ids, x.topk_weights)
    rows = _rand_expert_rows(m, s.h, 8)
    assert np.array_equal(ref.combine(m, x.topk_weights, rows), ref.combine_pagemode(m, rows))


# ------------------------------------------- apply_router_weight_on_input

def test_weight_on_input_scaling_closed_forms():
    """prepare with apply_router_weight_on_input (top_k == 1): a1 * bf16(w), rounded
    to bf16. Powers of two scale exactly, -1 negates, and a weight that bf16 cannot
    hold is rounded to bf16 *before* the product (1 + 2^-10 becomes exactly 1)."""
    rng = np.random.default_rng(5)
    a = wl.f32_to_bf16_bits(rng.standard_normal((12, 96), dtype=np.float32))
    x = wl.bf16_bits_to_f32(a)
    for w, expect in [(0.5, x * 0.5), (1.0, x), (-1.0, -x), (0.125, x / 8), (4.0, x * 4),
                      (1.0 + 2.0 ** -10, x)]:
        got = ref.scale_input(a, np.full((12, 1), w, np.float32))
        assert np.array_equal(wl.bf16_bits_to_f32(got), expect), w
    # a general weight: one rounding of the exact product (bf16 x bf16 fits in fp32)
    w = rng.random((12, 1), dtype=np.float32) + 0.1
    wb = wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(w))
    exact = x.astype(np.float64) * wb.astype(np.float64)
    got = wl.bf16_bits_to_f32(ref.scale_input(a, w)).astype(np.float64)
    assert np.all(np.abs(got - exact) <= 2.0 ** -8 * np.abs(exact))


# --------------------------------------------------- all-gather / reduce-scatter

@pytest.mark.parametrize("cfg,T", [(1, None), (2, 24), (5, 8)])
def test_agrs_route_equals_two_stage_combine_of_the_all_to_all_route(cfg, T):
    """Two different routes, written independently (rank-major loops over every
    gathered token vs per-slot partials of the dispatched rows), give the same bits
    with identity experts: each is a bf16 partial per destination rank summed over
    ranks in ascending order."""
    x = wl.make(wl.spec(cfg, T=T) if T else wl.spec(cfg))
    s = x.spec
    m = ref.dispatch_meta(s.W, s.E, s.K, s.T, x.topk_ids, x.topk_weights, x.num_tokens)
    rows = ref.dispatch_rows(m, x.a1)
    for f32 in (False, True):
        agrs, err = ref.agrs(s.W, s.E, s.K, s.T, x.a1, x.topk_ids, x.topk_weights, x.num_tokens, f32)
        assert err == 0
        assert np.array_equal(agrs, ref.combine_pagemode(m, rows, out_f32=f32))


def test_agrs_one_rank_is_the_single_fold():
    x = wl.make(wl.spec(2, W=1, E=8, T=40))
    s = x.spec
    m = ref.dispatch_meta(s.W, s.E, s.K, s.T, x.topk_ids, x.topk_weights)
    rows = ref.dispatch_rows(m, x.a1)
    agrs, _ = ref.agrs(s.W, s.E, s.K, s.T, x.a1, x.topk_ids, x.topk_weights)
    assert np.array_equal(agrs, ref.combine(m, x.topk_weights, rows))
    # identity experts with weights summing to one reproduce a1 on routed tokens
    routed = (x.topk_ids.reshape(-1, s.K) >= 0).any(axis=1)
    assert np.array_equal(agrs[routed], x.a1.reshape(-1, s.h)[routed])


def test_agrs_drops_bad_pairs_like_the_router():
    W, E, K, T = 2, 4, 3, 2
    ids = np.array([[[0, 9, -3], [1, 1, 2]], [[-1, -1, -1], [3, 0, -2]]], np.int32)
    w = np.full((W, T, K), 0.25, np.float32)
    a1 = wl.f32_to_bf16_bits(np.random.default_rng(1).standard_normal((W, T, 16), dtype=np.float32))
    out, err = ref.agrs(W, E, K, T, a1, ids, w, out_f32=True)
    assert err & ref.ERR_EXPERT_ID and err & ref.ERR_DUPLICATE
    x = wl.bf16_bits_to_f32(a1).reshape(W * T, 16)
    # token (0,0): only id 0 kept -> 0.25 x; token (0,1): ids 1 and 2 kept (on ranks 0 and 1)
    assert np.array_equal(out[0], wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(0.25 * x[0])))
    assert (out[2] == 0).all()


def test_agrs_worked_example_by_hand():
    """tests/golden/agrs_worked_example.json: a token whose three experts live on
    three ranks. The per-rank bf16 outputs summed in rank order round twice on
    ties (to even) and land one bf16 step below the single fp32 fold."""
    g = json.load(open(os.path.join(os.path.dirname(GOLDEN), "agrs_worked_example.json")))
    W, E, K, Tm, h = g["W"], g["E"], g["top_k"], g["max_tokens"], g["hidden"]
    a1 = np.zeros((W, Tm, h), np.float32)
    a1[0, 0] = g["a1"]
    ids = np.full((W, Tm, K), -1, np.int32)
    w = np.zeros((W, Tm, K), np.float32)
    for r in range(W):
        if g["topk_ids"][r]:
            ids[r, 0] = g["topk_ids"][r]
            w[r, 0] = g["topk_weights"][r]
    nt = np.array(g["num_tokens"], np.int32)
    x = wl.f32_to_bf16_bits(a1)
    out, err = ref.agrs(W, E, K, Tm, x, ids, w, nt, out_f32=False)
    assert err == 0
    assert np.array_equal(wl.bf16_bits_to_f32(out).reshape(W, h), np.array(g["expect_bf16_out"], np.float32))
    out32, _ = ref.agrs(W, E, K, Tm, x, ids, w, nt, out_f32=True)
    assert np.array_equal(out32.reshape(W, h), np.array(g["expect_f32_out"], np.float32))
    # the all-to-all route: single fold, and the page's two-stage rounding (= this route)
    m = ref.dispatch_meta(W, E, K, Tm, ids, w, nt)
    rows = ref.dispatch_rows(m, x)
    single = wl.bf16_bits_to_f32(ref.combine(m, w, rows)).reshape(W, h)
    assert np.array_equal(single[0], np.array(g["expect_single_fold_bf16"], np.float32))
    assert np.array_equal(ref.combine_pagemode(m, rows), out)


# ------------------------------------------- rounding of the combine fold, by hand

def _fold_golden():
    g = json.load(open(os.path.join(os.path.dirname(GOLDEN), "fold_rounding.json")))
    W, E, K, Tm, h = g["W"], g["E"], g["K"], g["Tm"], g["h"]
    ids = np.array(g["topk_ids"], np.int32)
    w = np.array(g["topk_weights"], np.float64)
    assert np.array_equal(w.astype(np.float32).astype(np.float64), w), "weights not fp32-exact"
    a1f = np.array(g["a1"], np.float32)
    a1 = wl.f32_to_bf16_bits(a1f)
    assert np.array_equal(wl.bf16_bits_to_f32(a1), a1f), "a1 not bf16-exact"
    nt = np.array(g["num_tokens"], np.int32)
    expect = np.array(g["expect_out"], np.float32).reshape(W * Tm, h)
    return g, W, E, K, Tm, h, ids, w.astype(np.float32), a1, nt, expect


def _same_bits(got, expect):
    got = np.asarray(got, np.float32)
    return np.array_equal(got.view(np.uint32), expect.view(np.uint32))


def test_fold_rounds_each_product_before_its_sum():
    """tests/golden/fold_rounding.json: the page's finalize forms the weighted rows
    as an fp32 tensor of their own and then accumulates them, so each product is
    rounded before it is added. Hand-derived dyadic cases where a fused
    multiply-add gives 2^-30 (or -2^-23, or one ulp more) instead of the separate
    roundings' result, and one where the fold order shows; checked on the single
    fold (both output types), the page's two-stage form and the all-gather /
    reduce-scatter route, all with identity experts."""
    g, W, E, K, Tm, h, ids, w, a1, nt, expect = _fold_golden()
    m = ref.dispatch_meta(W, E, K, Tm, ids, w, nt)
    assert m.err == 0
    rows = ref.dispatch_rows(m, a1)        # identity experts: each pair's row is its token
    out32 = ref.combine(m, w, rows, out_f32=True)
    assert _same_bits(out32, expect), out32
    outb = ref.combine(m, w, rows, out_f32=False)
    assert _same_bits(wl.bf16_bits_to_f32(outb), expect)
    for f32 in (False, True):
        page = ref.combine_pagemode(m, rows, out_f32=f32)
        page = page if f32 else wl.bf16_bits_to_f32(page)
        assert _same_bits(page, expect), (f32, page)
        ag, err = ref.agrs(W, E, K, Tm, a1, ids, w, nt, out_f32=f32)
        assert err == 0
        ag = ag if f32 else wl.bf16_bits_to_f32(ag)
        assert _same_bits(ag, expect), (f32, ag)
