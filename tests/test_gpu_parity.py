"""GPU parity: the sm_103a path through the C-ABI against the CPU oracle.

Dispatch outputs (expert_num_tokens, slot counts, combine map, received
metadata, payload bytes of every delivered row) must match bit for bit;
combine must stay within 1e-2 (bf16 out) / 1e-5 (fp32 out) max relative error
and, since the kernel folds in the oracle's order, is also checked for
identical bits. All five named workloads run at full size in the launch
configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

from combine_ep_route_gb300 import EpConfig, EpContext, EpError, workloads as wl
from combine_ep_route_gb300 import _lib as L
from oracle import ref
from tests import _gpu_harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def _roundtrip(x, dev, path="fused", out_f32=(False,), seed=1, ctx_kw=None, opts=None):
    ctx = H.make_ctx(x, dev, **(ctx_kw or {}))
    for k, v in (opts or {}).items():
        ctx.set_option(k, v)
    a1, ids, w, nt, extras = H.inputs_dev(x, dev)
    out = ctx.dispatch(a1, ids, w, num_tokens=nt, extras=extras, path=path)
    ctx.check()
    m = H.oracle_meta(x)
    assert m.err == 0
    H.check_meta(ctx, m, x, out.expert_num_tokens)
    H.check_rows(out, m, x, a1, extras)
    for i, f32 in enumerate(out_f32):
        if i:   # combine again needs a fresh dispatch (the state rule)
            ctx.dispatch(a1, ids, w, num_tokens=nt, extras=extras, out=out, path=path)
            ctx.check()
        packed = H.fill_pool_rows(out, m, x.spec.h, seed)
        H.check_combine(ctx, out.b_a1, m, x, packed, f32)
    return ctx, out, m


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_named_workload_full_size(dev, cfg):
    x = wl.make(cfg)
    _roundtrip(x, dev, out_f32=(False, True) if cfg in (1, 3) else (False,))


@pytest.mark.parametrize("cfg", [1, 2])
def test_identity_experts_reproduce_a1(dev, cfg):
    x = wl.make(cfg)
    s = x.spec
    ctx = H.make_ctx(x, dev)
    a1, ids, w, nt, extras = H.inputs_dev(x, dev)
    out = ctx.dispatch(a1, ids, w, extras=extras)
    y = ctx.combine(out.b_a1)
    ctx.check()
    routed = (x.topk_ids >= 0).any(axis=2)
    got = H.bits_host(y).reshape(s.W, s.T, s.h)
    assert np.array_equal(got[routed], x.a1[routed])
    assert (got[~routed] == 0).all()


@pytest.mark.parametrize("cfg,T", [(1, None), (2, None), (4, 96), (5, 40)])
def test_sendbuf_path_matches_oracle_and_fused(dev, cfg, T):
    x = wl.make(wl.spec(cfg, T=T) if T else wl.spec(cfg))
    s = x.spec
    ctx, out, m = _roundtrip(x, dev, path="sendbuf", ctx_kw=dict(sendbuf=True))
    # send and receive rank blocks hold the oracle's packed and exchanged rows
    md = ctx.metadata()
    src = np.concatenate([x.a1.view(np.uint8).reshape(s.W, s.T, -1)] + x.extras, axis=2)
    rb = src.shape[2]
    send_x = np.zeros((s.W, s.W, s.T, rb), np.uint8)
    ref.lib().oracle_pack(s.W, s.T, rb, m.send_cnt.ctypes.data, m.send_tok.ctypes.data,
                          src.ctypes.data, send_x.ctypes.data)
    recv_x = np.zeros_like(send_x)
    ref.lib().oracle_exchange(s.W, s.T, rb, send_x.ctypes.data, recv_x.ctypes.data)
    vs = np.arange(s.T)[None, None, :] < m.send_cnt[:, :, None]
    vr = np.arange(s.T)[None, None, :] < m.recv_cnt[:, :, None]
    assert np.array_equal(md["send_x"].cpu().numpy()[vs], send_x[vs])
    assert np.array_equal(md["recv_x"].cpu().numpy()[vr], recv_x[vr])
    # and the fused path delivers the same bytes
    ctx2 = H.make_ctx(x, dev)
    a1, ids, w, nt, extras = H.inputs_dev(x, dev)
    out2 = ctx2.dispatch(a1, ids, w, num_tokens=nt, extras=extras)
    ctx2.check()
    H.check_rows(out2, m, x, a1, extras)


def _custom(W, E, K, T, h, seed=0, pad=0.0, extras=(), num_tokens=None):
    s = wl.WorkloadSpec(f"w{W}-e{E}-k{K}-t{T}-h{h}", W=W, E=E, K=K, T=T, h=h, pad_frac=pad,
                        extra_f32_cols=tuple(extras), seed=seed)
    return wl.make(s, num_tokens=num_tokens)


@pytest.mark.parametrize("W,E,K,T,h,pad,extras", [
    (1, 6, 3, 50, 64, 0.1, ()),            # one rank: a counting sort by expert
    (4, 8, 4, 33, 32, 0.0, ()),            # K > e_local: two slots per token
    (3, 12, 2, 300, 8, 0.2, (4,)),         # two routing tiles per rank, ragged tail, 16-B rows
    (2, 4, 2, 1, 16, 0.0, ()),             # one token per rank
    (64, 1024, 16, 20, 64, 0.1, (4, 12)),  # the library's limits on W, E, top_k; two extras
    (8, 64, 8, 700, 2048, 0.05, ()),       # 3 tiles per rank
    (4, 32, 6, 150, 5120, 0.05, (16,)),    # 10 KiB rows in five 2 KiB units, top_k 6
    (8, 64, 8, 90, 1536, 0.0, ()),         # 3 KiB rows, moved whole
])
def test_edge_shapes(dev, W, E, K, T, h, pad, extras):
    _roundtrip(_custom(W, E, K, T, h, seed=W + E + T, pad=pad, extras=extras), dev, out_f32=(False, True))


def _same_ids(W, E, K, T, h, row_ids, seed):
    """Every token of every rank chooses the same experts (degenerate routing)."""
    x = _custom(W, E, K, T, h, seed=seed)
    x.topk_ids[:] = np.asarray(row_ids, np.int32)[None, None, :]
    return x


@pytest.mark.parametrize("path", ["fused", "sendbuf"])
def test_one_expert_set_filled_to_capacity(dev, path):
    """All tokens pick experts 0..3, all on rank 0: each of those experts receives
    W * max_tokens rows, exactly its capacity, and every other rank receives none."""
    W, E, K, T, h = 4, 16, 4, 200, 256
    x = _same_ids(W, E, K, T, h, [0, 1, 2, 3], seed=11)
    ctx, out, m = _roundtrip(x, dev, path=path, out_f32=(False, True),
                             ctx_kw=dict(sendbuf=path == "sendbuf"))
    ent = out.expert_num_tokens.cpu().numpy().reshape(W, E // W)
    assert (ent[0] == W * T).all() and (ent[1:] == 0).all()
    _check_two_stage(x, dev)


def test_every_token_reaches_every_rank(dev):
    """One expert per rank for every token (top_k = W): every token is sent to every
    destination, so each (source, destination) block holds all T slots."""
    W, E, K, T, h = 8, 64, 8, 130, 512
    x = _same_ids(W, E, K, T, h, [d * 8 + (5 * d) % 8 for d in range(8)][::-1], seed=12)
    ctx, out, m = _roundtrip(x, dev, out_f32=(False, True))
    assert (m.send_cnt == T).all()
    _check_two_stage(x, dev)


def test_side_streams_and_two_contexts(dev):
    """Dispatch and combine are enqueued on the caller's current stream: two
    contexts on two side streams, launched interleaved with no synchronisation
    between them, each match the oracle (combine on identity experts)."""
    xa = wl.make(2)
    xb = _custom(4, 32, 4, 150, 1024, seed=21, pad=0.1)
    streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    runs = []
    for x, st in zip((xa, xb), streams):
        with torch.cuda.stream(st):
            ctx = H.make_ctx(x, dev)
            a1, ids, w, nt, extras = H.inputs_dev(x, dev)
            out = ctx.dispatch(a1, ids, w, num_tokens=nt, extras=extras)
        runs.append((x, ctx, out, a1, extras))
    ys = []
    for (x, ctx, out, a1, extras), st in zip(runs, streams):
        with torch.cuda.stream(st):
            ys.append(ctx.combine(out.b_a1))
    torch.cuda.synchronize(dev)
    for (x, ctx, out, a1, extras), y in zip(runs, ys):
        ctx.check()
        m = H.oracle_meta(x)
        H.check_meta(ctx, m, x, out.expert_num_tokens)
        H.check_rows(out, m, x, a1, extras)
        exp = ref.combine(m, x.topk_weights, ref.dispatch_rows(m, x.a1))
        assert np.array_equal(H.bits_host(y).reshape(exp.shape), exp)


def test_ragged_and_empty_ranks(dev):
    nt = np.array([0, 17, 128, 3, 64, 0, 127, 1], np.int32)
    x = _custom(8, 64, 8, 128, 256, seed=4, pad=0.05, num_tokens=nt)
    _roundtrip(x, dev, out_f32=(False, True))
    # every id -1: nothing is sent, nothing delivered, all outputs zero
    x0 = _custom(4, 16, 4, 40, 64, seed=5)
    x0.topk_ids[:] = -1
    ctx, out, m = _roundtrip(x0, dev)
    assert int(out.expert_num_tokens.sum()) == 0


def test_zero_pad_flag(dev):
    x = wl.make(wl.spec(2, T=32))
    s = x.spec
    ctx = H.make_ctx(x, dev, zero_pad=True)
    a1, ids, w, nt, extras = H.inputs_dev(x, dev)
    out = ctx.alloc_dispatch_outputs()
    out.b_a1.fill_(3.0)
    ctx.dispatch(a1, ids, w, out=out)
    ctx.check()
    m = H.oracle_meta(x)
    H.check_rows(out, m, x, a1, extras)
    b = out.b_a1.view(s.E, -1, s.h)
    for e in range(s.E):
        n = int(m.expert_num_tokens.reshape(-1)[e])
        assert (b[e, n:] == 0).all()
    # received-slot metadata past the counts carries the page's fill values
    md = ctx.metadata()
    assert np.array_equal(md["recv_eloc"].cpu().numpy(), m.recv_eloc)
    assert np.array_equal(md["recv_w"].cpu().numpy(), m.recv_w)
    assert np.array_equal(md["recv_row"].cpu().numpy(), H.expected_recv_row(m))


def test_device_errors_are_reported_and_pairs_dropped(dev):
    x = _custom(4, 16, 4, 64, 64, seed=9)
    x.topk_ids[0, 3, 1] = 16            # id >= E
    x.topk_ids[2, 5, 3] = x.topk_ids[2, 5, 0]   # repeated id
    ctx = H.make_ctx(x, dev)
    a1, ids, w, nt, extras = H.inputs_dev(x, dev)
    out = ctx.dispatch(a1, ids, w)
    st = ctx.status()
    assert st in (L.EP_ERR_EXPERT_ID, L.EP_ERR_DUPLICATE)
    m = H.oracle_meta(x)
    assert m.err & ref.ERR_EXPERT_ID and m.err & ref.ERR_DUPLICATE
    H.check_meta(ctx, m, x, out.expert_num_tokens)
    H.check_rows(out, m, x, a1, extras)
    ctx.combine(out.b_a1)
    assert ctx.status() == 0
    # num_tokens above max_tokens
    bad = torch.tensor([64, 65, 0, 1], dtype=torch.int32, device=dev)
    ctx.dispatch(a1, ids, w, num_tokens=bad)
    assert ctx.status() == L.EP_ERR_CAPACITY
    ctx.reset()


def test_state_rule(dev):
    x = wl.make(1)
    ctx = H.make_ctx(x, dev)
    a1, ids, w, nt, extras = H.inputs_dev(x, dev)
    out = ctx.dispatch(a1, ids, w)
    with pytest.raises(EpError) as e:
        ctx.dispatch(a1, ids, w)
    assert e.value.code == L.EP_ERR_STATE
    ctx.combine(out.b_a1)
    with pytest.raises(EpError) as e:
        ctx.combine(out.b_a1)
    assert e.value.code == L.EP_ERR_STATE
    ctx.check()


def test_wait_limit_reports_timeout_then_recovers(dev):
    """A routing tile that never publishes (test hook) makes its successors'
    bounded waits run out: the call reports EP_ERR_TIMEOUT and the next
    dispatch on the same context is correct again."""
    x = _custom(2, 8, 2, 1024, 64, seed=3)      # 16 routing tiles per rank
    ctx = H.make_ctx(x, dev)
    ctx.set_option(L.EP_OPT_SMALL_DISPATCH, 0)   # the tiled routing, whose tiles wait on each other
    ctx.set_option(L.EP_OPT_WAIT_LIMIT_NS, 20_000_000)
    ctx.set_option(L.EP_OPT_FAULT_SKIP_PUBLISH, 2)
    a1, ids, w, nt, extras = H.inputs_dev(x, dev)
    out = ctx.dispatch(a1, ids, w)
    assert ctx.status() == L.EP_ERR_TIMEOUT
    ctx.reset()
    ctx.set_option(L.EP_OPT_FAULT_SKIP_PUBLISH, -1)
    out = ctx.dispatch(a1, ids, w)
    ctx.check()
    m = H.oracle_meta(x)
    H.check_meta(ctx, m, x, out.expert_num_tokens)
    H.check_rows(out, m, x, a1, extras)


@pytest.mark.parametrize("opts", [
    {L.EP_OPT_PDL: 0},
    {L.EP_OPT_MOVE_PIPES: 1},
    {L.EP_OPT_MOVE_PIPES: 8, L.EP_OPT_MOVE_CTAS_PER_SM: 2},
    {L.EP_OPT_KERNEL_TIMING: 1, L.EP_OPT_COMBINE_CTAS_PER_SM: 2},
    {L.EP_OPT_MOVE_CHUNK_BYTES: 2048, L.EP_OPT_MOVE_MAX_STAGES: 16},
    {L.EP_OPT_MOVE_CHUNK_BYTES: 1024, L.EP_OPT_MOVE_MAX_STAGES: 2, L.EP_OPT_MOVE_PIPES: 2},
    {L.EP_OPT_MOVE_CHUNK_BYTES: 0},
    {L.EP_OPT_FUSED_DISPATCH: 0},
    {L.EP_OPT_FUSED_DISPATCH: 0, L.EP_OPT_PDL: 1},
    {L.EP_OPT_ROUTE_CTAS: 1},
    {L.EP_OPT_ROUTE_CTAS: 3, L.EP_OPT_MOVE_PIPES: 4},
    {L.EP_OPT_ROUTE_CTAS: 4096},
    {L.EP_OPT_ROUTE_CTAS: 0},
    {L.EP_OPT_SMALL_DISPATCH: -1},
    {L.EP_OPT_SMALL_DISPATCH: 1, L.EP_OPT_KERNEL_TIMING: 1},
    {L.EP_OPT_SMALL_DISPATCH: 1, L.EP_OPT_PDL: 1},
])
@pytest.mark.parametrize("path", ["fused", "sendbuf"])
def test_launch_options_do_not_change_results(dev, opts, path):
    x = wl.make(wl.spec(4, T=128))   # 8 KiB rows plus a 128-byte extra payload
    # a batch this small takes the small-batch dispatch unless it is turned off;
    # the other options shape the tiled one-launch dispatch
    _roundtrip(x, dev, opts={L.EP_OPT_SMALL_DISPATCH: 0, **opts}, path=path,
               ctx_kw=dict(sendbuf=path == "sendbuf"))


# 32 routing tiles (every CTA routes) and 96 (32 elected routers); at T = 64 also
# the small-batch dispatch
@pytest.mark.parametrize("T,small", [(64, 0), (64, -1), (160, -1)])
def test_repeated_steps_are_identical(dev, T, small):
    x = wl.make(wl.spec(5, T=T))
    ctx = H.make_ctx(x, dev)
    ctx.set_option(L.EP_OPT_SMALL_DISPATCH, small)
    a1, ids, w, nt, extras = H.inputs_dev(x, dev)
    outs = []
    for _ in range(4):
        d = ctx.dispatch(a1, ids, w, num_tokens=nt)
        outs.append((d.expert_num_tokens.clone(), ctx.combine(d.b_a1).clone()))
    ctx.check()
    for a, b in outs[1:]:
        assert torch.equal(a, outs[0][0]) and torch.equal(b.view(torch.int16), outs[0][1].view(torch.int16))


def _check_two_stage(x, dev):
    s = x.spec
    ctx = H.make_ctx(x, dev, sendbuf=True)
    a1, ids, w, nt, extras = H.inputs_dev(x, dev)
    m = H.oracle_meta(x)
    for f32 in (False, True):
        out = ctx.dispatch(a1, ids, w, num_tokens=nt, extras=extras)
        ctx.check()
        packed = H.fill_pool_rows(out, m, s.h, 3)
        got = ctx.combine_two_stage(out.b_a1, out_dtype=torch.float32 if f32 else torch.bfloat16)
        ctx.check()
        exp = ref.combine_pagemode(m, packed, out_f32=f32)
        if f32:
            g = got.cpu().numpy().reshape(-1, s.h)
        else:
            g = H.bits_host(got).reshape(-1, s.h)
        assert np.array_equal(g, exp), "two-stage combine differs from the page-mode oracle"
        single = ref.combine(m, x.topk_weights, packed, out_f32=f32)
        gf = g if f32 else wl.bf16_bits_to_f32(g)
        sf = single if f32 else wl.bf16_bits_to_f32(single)
        assert np.linalg.norm(gf.astype(np.float64) - sf) <= 1e-2 * np.linalg.norm(sf)


@pytest.mark.parametrize("cfg,T", [(1, None), (2, None), (3, 128), (4, 96), (5, 40)])
def test_two_stage_combine_matches_page_mode_oracle(dev, cfg, T):
    """ep_combine_two_stage restates the page's own finalize (bf16 per-rank partials,
    summed over ranks in the output type): bit-identical to the oracle's page-mode
    combine, and within the page's bound of the single-rounding fold."""
    _check_two_stage(wl.make(wl.spec(cfg, T=T) if T else wl.spec(cfg)), dev)


@pytest.mark.parametrize("W,E,K,T,h,pad", [
    (64, 1024, 16, 20, 64, 0.1),   # top_k 16: sixteen send rows per token to order, wide slots
    (4, 8, 4, 33, 32, 0.0),        # top_k > e_local: two columns in every slot
    (1, 6, 3, 50, 64, 0.1),        # one rank
    (3, 12, 2, 300, 8, 0.2),       # two routing tiles per rank, ragged tail, 16-byte rows
])
def test_two_stage_combine_edge_shapes(dev, W, E, K, T, h, pad):
    _check_two_stage(_custom(W, E, K, T, h, seed=3 * W + E + T, pad=pad), dev)


@pytest.mark.parametrize("path", ["fused", "sendbuf"])
def test_weight_on_input_top1(dev, path):
    """apply_router_weight_on_input: rows arrive as bf16(a1 * bf16(w)) and combine
    carries unit weights (vLLM AllToAllBatchedPrepareAndFinalize.prepare)."""
    x = _custom(8, 64, 1, 256, 2048, seed=21, pad=0.05, extras=(4,))
    s = x.spec
    ctx = H.make_ctx(x, dev, sendbuf=path == "sendbuf", weight_on_input=True)
    a1, ids, w, nt, extras = H.inputs_dev(x, dev)
    out = ctx.dispatch(a1, ids, w, num_tokens=nt, extras=extras, path=path)
    ctx.check()
    ones = np.ones_like(x.topk_weights)
    m = ref.dispatch_meta(s.W, s.E, s.K, s.T, x.topk_ids, ones, x.num_tokens)
    H.check_meta(ctx, m, wl.Workload(x.spec, x.a1, x.topk_ids, ones, x.num_tokens, x.extras),
                 out.expert_num_tokens)
    scaled = ref.scale_input(x.a1, x.topk_weights)
    H.check_rows(out, m, x, H.bf16_dev(scaled, dev), extras)
    y = ctx.combine(out.b_a1)
    ctx.check()
    exp = ref.combine(m, ones, ref.dispatch_rows(m, scaled))
    assert np.array_equal(H.bits_host(y).reshape(-1, s.h), exp)


@pytest.mark.parametrize("T", [64, 160])
def test_graph_replay_on_new_inputs(dev, T):
    """A dispatch + combine captured once in a CUDA graph and replayed on new
    inputs copied into the same buffers stays exact: the routing look-back epoch
    and the launch's counters (tickets, routers, units) are rearmed on the device,
    so no host call is needed between replays."""
    xs = [wl.make(wl.spec(5, T=T), seed=s) for s in (11, 12, 13)]
    x0 = xs[0]
    s = x0.spec
    ctx = H.make_ctx(x0, dev)
    a1, ids, w, nt, extras = H.inputs_dev(x0, dev)
    out = ctx.alloc_dispatch_outputs()
    y = torch.empty((s.W, s.T, s.h), dtype=torch.bfloat16, device=dev)
    ctx.dispatch(a1, ids, w, num_tokens=nt, out=out)   # first use initialises the workspace
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
        assert ctx.status() == 0
        m = H.oracle_meta(x)
        assert np.array_equal(out.expert_num_tokens.cpu().numpy(), m.expert_num_tokens)
        H.check_rows(out, m, x, a1, [])
        exp = ref.combine(m, x.topk_weights, ref.dispatch_rows(m, x.a1))
        assert np.array_equal(H.bits_host(y).reshape(-1, s.h), exp)


@pytest.mark.parametrize("x_dtype,extra_cols", [("fp8", 56), ("fp4x2", 112)])
@pytest.mark.parametrize("path", ["fused", "sendbuf"])
def test_quantised_payload_rows(dev, x_dtype, extra_cols, path):
    """Quantised activations as the page's one-sided sizing assumes (fp8 rows of h
    bytes with fp32 block scales, or packed fp4 rows of h/2 bytes with 4-byte scale
    words) travel as opaque bytes; rows and scales land byte-exact, and combine
    still reduces bf16 expert outputs."""
    base = wl.make(wl.spec(3, T=64))
    s = base.spec
    rng = np.random.default_rng(17)
    row_bytes = s.h if x_dtype == "fp8" else s.h // 2
    a1_bytes = rng.integers(0, 256, size=(s.W, s.T, row_bytes), dtype=np.uint8)
    scales = rng.integers(0, 256, size=(s.W, s.T, extra_cols * 4), dtype=np.uint8)
    from combine_ep_route_gb300 import EpConfig, EpContext
    cfg = EpConfig(s.W, s.E, s.K, s.T, s.h, extra_row_bytes=(extra_cols * 4,), sendbuf=path == "sendbuf",
                   x_dtype=x_dtype)
    ctx = EpContext(cfg, dev)
    a1 = torch.from_numpy(a1_bytes).to(dev).view(cfg.x_torch_dtype)
    ids = torch.from_numpy(base.topk_ids).to(dev)
    w = torch.from_numpy(base.topk_weights).to(dev)
    ex = [torch.from_numpy(scales).to(dev)]
    out = ctx.dispatch(a1, ids, w, extras=ex, path=path)
    ctx.check()
    m = H.oracle_meta(base)
    rows = ref.dispatch_rows(m, np.concatenate([a1_bytes, scales], axis=2))
    flat, _ = H.valid_rows(m)
    fi = torch.from_numpy(flat).to(dev)
    got = out.b_a1.view(torch.uint8).view(-1, row_bytes).index_select(0, fi).cpu().numpy()
    assert np.array_equal(got, rows[:, :row_bytes])
    got_sc = out.extra_out[0].view(-1, extra_cols * 4).index_select(0, fi).cpu().numpy()
    assert np.array_equal(got_sc, rows[:, row_bytes:])
    # combine on bf16 expert outputs of the delivered rows
    expert_out = torch.zeros((s.W, s.E // s.W, ctx.expert_cap, s.h), dtype=torch.bfloat16, device=dev)
    holder = type("O", (), {})()
    holder.b_a1 = expert_out
    packed = H.fill_pool_rows(holder, m, s.h, 6)
    y = ctx.combine(expert_out)
    ctx.check()
    exp = ref.combine(m, base.topk_weights, packed)
    assert np.array_equal(H.bits_host(y).reshape(-1, s.h), exp)
