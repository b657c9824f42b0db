"""GPU parity of the small-batch dispatch (every CTA counts its own prefix from
the earlier tokens' ids; no waits between CTAs) against the oracle, and against
the tiled one-launch dispatch on the same inputs.

The shapes cover one token per CTA, CTAs that straddle a rank boundary, 32
token slots per CTA (the most it takes), the library's W / E / top_k limits,
ragged and empty ranks, extra payloads, quantised rows and the device-side
error paths (bad ids, repeated ids, token counts out of range).
"""
import numpy as np
import pytest
import torch

from combine_ep_route_gb300 import EpConfig, EpContext, workloads as wl
from combine_ep_route_gb300 import _lib as L
from oracle import ref
from tests import _gpu_harness as H
from tests.test_gpu_parity import _custom

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def _run(x, dev, small, expect_status=0, out_f32=False, seed=4):
    """Dispatch (+ combine) with the small-batch dispatch on (-1) or off (0);
    checks which kernel ran and every output against the oracle."""
    ctx = H.make_ctx(x, dev)
    ctx.set_option(L.EP_OPT_SMALL_DISPATCH, small)
    ctx.kernel_times()
    a1, ids, w, nt, extras = H.inputs_dev(x, dev)
    out = ctx.dispatch(a1, ids, w, num_tokens=nt, extras=extras)
    assert ctx.status() == expect_status
    kt = ctx.kernel_times()
    ran_small = kt["dispatch_small"][0] == 1
    assert ran_small == (small != 0), kt
    s = x.spec
    m = ref.dispatch_meta(s.W, s.E, s.K, s.T, x.topk_ids, x.topk_weights, x.num_tokens)
    H.check_meta(ctx, m, x, out.expert_num_tokens)
    H.check_rows(out, m, x, a1, extras)
    packed = H.fill_pool_rows(out, m, s.h, seed)
    H.check_combine(ctx, out.b_a1, m, x, packed, out_f32)
    return ctx, out, m


@pytest.mark.parametrize("cfg", [1, 2])
def test_named_small_workloads(dev, cfg):
    x = wl.make(cfg)
    for small in (-1, 0):
        for f32 in (False, True):
            _run(x, dev, small, out_f32=f32)


@pytest.mark.parametrize("W,E,K,T,h,pad,extras", [
    (3, 12, 2, 301, 8, 0.2, (4,)),         # CTAs straddle rank boundaries, 16-byte rows
    (64, 1024, 16, 16, 64, 0.1, (4, 12)),  # W, E and top_k at the library's limits; 16384 ids
    (16, 32, 2, 1, 128, 0.0, ()),          # one token per rank and per CTA
    (8, 24, 3, 608, 64, 0.05, ()),         # 32 token slots per CTA
    (4, 8, 8, 40, 256, 0.0, ()),           # top_k > e_local: two slots per token
    (1, 6, 3, 50, 64, 0.1, ()),            # one rank: a counting sort by expert
    (8, 64, 8, 128, 5120, 0.05, (16,)),    # 10 KiB rows with an extra payload
    (4, 8, 1, 100, 64, 0.1, ()),           # top_k 1
    (8, 8, 5, 60, 64, 0.0, (4,)),          # one expert per rank, top_k 5 (not a power of two)
])
def test_small_edge_shapes_match_oracle_and_tiled_path(dev, W, E, K, T, h, pad, extras):
    x = _custom(W, E, K, T, h, seed=W * 7 + T, pad=pad, extras=extras)
    _, o_small, _ = _run(x, dev, -1)
    b_small = o_small.b_a1.clone()
    _, o_tiled, m = _run(x, dev, 0)
    flat, _ = H.valid_rows(m)
    fi = torch.from_numpy(flat).to(dev)
    assert torch.equal(b_small.view(-1, h).view(torch.int16).index_select(0, fi),
                       o_tiled.b_a1.view(-1, h).view(torch.int16).index_select(0, fi))


def test_ragged_and_empty_ranks(dev):
    nt = np.array([128, 0, 37, 128, 1, 0, 64, 127], np.int32)
    x = wl.make(wl.spec(2), num_tokens=nt)
    _run(x, dev, -1)


def test_device_errors_match_the_tiled_path(dev):
    """Bad ids and repeated ids are reported and dropped exactly as the tiled
    routing does; a token count above max_tokens is clamped and reported."""
    x = wl.make(wl.spec(2, T=64))
    x.topk_ids[0, 3, 2] = 1000            # >= E: dropped, EP_ERR_EXPERT_ID
    _run(x, dev, -1, expect_status=L.EP_ERR_EXPERT_ID)
    y = wl.make(wl.spec(2, T=64))
    t = int(np.nonzero((y.topk_ids[5, :] >= 0).all(axis=1))[0][0])
    y.topk_ids[5, t, 4] = y.topk_ids[5, t, 0]   # a repeat: the later one dropped
    _run(y, dev, -1, expect_status=L.EP_ERR_DUPLICATE)
    # num_tokens above max_tokens: clamped to max_tokens and reported
    z = wl.make(wl.spec(2, T=64))
    s = z.spec
    ctx = H.make_ctx(z, dev)
    a1, ids, w, nt, extras = H.inputs_dev(z, dev)
    nt[3] = s.T + 5
    out = ctx.dispatch(a1, ids, w, num_tokens=nt)
    assert ctx.status() == L.EP_ERR_CAPACITY
    m = ref.dispatch_meta(s.W, s.E, s.K, s.T, z.topk_ids, z.topk_weights, z.num_tokens)
    H.check_meta(ctx, m, z, out.expert_num_tokens)


@pytest.mark.parametrize("x_dtype", ["fp8", "fp4x2"])
def test_quantised_rows(dev, x_dtype):
    x = wl.make(wl.spec(2, T=64))
    s = x.spec
    rb = s.h if x_dtype == "fp8" else s.h // 2
    cfg = EpConfig(s.W, s.E, s.K, s.T, s.h, extra_row_bytes=(32,), x_dtype=x_dtype)
    ctx = EpContext(cfg, dev)
    ctx.kernel_times()
    rng = np.random.default_rng(3)
    rows = rng.integers(0, 256, size=(s.W, s.T, rb), dtype=np.uint8)
    scl = rng.integers(0, 256, size=(s.W, s.T, 32), dtype=np.uint8)
    a1 = torch.from_numpy(rows).to(dev).view(cfg.x_torch_dtype)
    ids = torch.from_numpy(x.topk_ids).to(dev)
    w = torch.from_numpy(x.topk_weights).to(dev)
    ex = torch.from_numpy(scl).to(dev)
    out = ctx.dispatch(a1, ids, w, extras=[ex])
    ctx.check()
    assert ctx.kernel_times()["dispatch_small"][0] == 1
    m = ref.dispatch_meta(s.W, s.E, s.K, s.T, x.topk_ids, x.topk_weights)
    want = ref.dispatch_rows(m, np.concatenate([rows, scl], axis=2))
    flat, _ = H.valid_rows(m)
    got_x = out.b_a1.view(torch.uint8).reshape(-1, rb).cpu().numpy()[flat]
    got_s = out.extra_out[0].reshape(-1, 32).cpu().numpy()[flat]
    assert np.array_equal(got_x, want[:, :rb]) and np.array_equal(got_s, want[:, rb:])


def test_graph_replay_and_repeats(dev):
    """Captured once, replayed on new inputs: the small-batch dispatch keeps no
    state between launches."""
    xs = [wl.make(wl.spec(2), seed=s) for s in (21, 22, 23)]
    s = xs[0].spec
    ctx = H.make_ctx(xs[0], dev)
    a1, ids, w, nt, extras = H.inputs_dev(xs[0], dev)
    out = ctx.alloc_dispatch_outputs()
    y = torch.empty((s.W, s.T, s.h), dtype=torch.bfloat16, device=dev)
    ctx.dispatch(a1, ids, w, num_tokens=nt, out=out)
    ctx.combine(out.b_a1, out=y)
    ctx.check()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ctx.dispatch(a1, ids, w, num_tokens=nt, out=out)
        ctx.combine(out.b_a1, out=y)
    for x in xs:
        a1n, idsn, wn, ntn, _ = H.inputs_dev(x, dev)
        a1.copy_(a1n)
        ids.copy_(idsn)
        w.copy_(wn)
        nt.copy_(ntn)
        g.replay()
        torch.cuda.synchronize()
        ctx.check()
        m = H.oracle_meta(x)
        H.check_meta(ctx, m, x, out.expert_num_tokens)
        H.check_rows(out, m, x, a1, extras)
        routed = (x.topk_ids >= 0).any(axis=2)
        got = H.bits_host(y).reshape(s.W, s.T, s.h)
        assert np.array_equal(got[routed], x.a1[routed])   # identity experts, weights sum to 1
