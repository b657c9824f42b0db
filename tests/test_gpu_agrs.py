"""GPU parity of the all-gather / reduce-scatter route (``ep_agrs``).

The gathered ids, weights and token rows must equal the inputs byte for byte
on every rank, and the reduce-scattered output must equal the oracle's bits
(it folds and sums in the oracle's order with the same roundings; the bf16 /
fp32 tolerances are checked as well). A second check runs the all-to-all
route on the GPU -- dispatch, identity experts, the page-rounding two-stage
combine -- and requires the same bits as this route.
"""
import numpy as np
import pytest
import torch

from combine_ep_route_gb300 import EpConfig, EpContext, agrs, alloc_agrs_buffers, workloads as wl
from combine_ep_route_gb300 import _lib as L
from oracle import ref
from tests import _gpu_harness as H
from tests._metrics import max_rel_err, TOL_BF16_OUT, TOL_F32_OUT

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def _cfg(s: wl.WorkloadSpec) -> EpConfig:
    return EpConfig(s.W, s.E, s.K, s.T, s.h)


def _run(x: wl.Workload, dev, out_f32: bool, buffers=None, nt_dev=True):
    s = x.spec
    a1, ids, w, nt, _ = H.inputs_dev(x, dev)
    buf = buffers if buffers is not None else alloc_agrs_buffers(_cfg(s), dev)
    out = agrs(_cfg(s), a1, ids, w, num_tokens=nt if nt_dev else None,
               out_dtype=torch.float32 if out_f32 else torch.bfloat16, buffers=buf)
    torch.cuda.synchronize(dev)
    return out, buf


def _host(out: torch.Tensor, out_f32: bool) -> np.ndarray:
    if out_f32:
        return out.cpu().numpy()
    return wl.bf16_bits_to_f32(H.bits_host(out))


def _compare(got: np.ndarray, exp: np.ndarray, out_f32: bool) -> None:
    e = exp if out_f32 else wl.bf16_bits_to_f32(exp)
    g = got.reshape(e.shape)
    err = max_rel_err(g, e)
    tol = TOL_F32_OUT if out_f32 else TOL_BF16_OUT
    assert err <= tol, f"max relative error {err} > {tol}"
    assert np.array_equal(g.view(np.uint32), e.view(np.uint32)), "not bit-identical to the oracle"


def _check_gather(buf, x: wl.Workload) -> None:
    s = x.spec
    valid = (np.arange(s.T)[None, :] < x.num_tokens[:, None]).reshape(-1)
    vi = torch.from_numpy(np.nonzero(valid)[0]).to(buf.x_g.device)
    a1 = x.a1.reshape(s.W * s.T, s.h)[valid]
    ids = x.topk_ids.reshape(-1, s.K)[valid]
    w = x.topk_weights.reshape(-1, s.K)[valid]
    for d in range(s.W):
        assert np.array_equal(H.bits_host(buf.x_g[d].index_select(0, vi)), a1), f"x_g of rank {d}"
        assert np.array_equal(buf.ids_g[d].index_select(0, vi).cpu().numpy(), ids), f"ids_g of rank {d}"
        assert np.array_equal(buf.w_g[d].index_select(0, vi).cpu().numpy(), w), f"w_g of rank {d}"


CASES = [
    (wl.spec(1), None),
    (wl.spec(2), None),
    (wl.spec(2), [128, 0, 77, 1, 128, 5, 64, 127]),   # ragged, one empty rank
    (wl.spec(4, T=40), None),                           # zipf ids, W=16
    (wl.spec(5, T=12), None),                           # grouped ids, padding rows, W=32
    (wl.spec(3, T=33), [33, 32, 1, 0, 17, 33, 2, 31]),  # h=7168, ragged tail
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_agrs_matches_oracle(dev, case):
    s, nt = CASES[case]
    x = wl.make(s, num_tokens=nt)
    for f32 in (False, True):
        out, buf = _run(x, dev, f32)
        assert int(buf.status.item()) == 0
        _check_gather(buf, x)
        exp, err = ref.agrs(s.W, s.E, s.K, s.T, x.a1, x.topk_ids, x.topk_weights, x.num_tokens, f32)
        assert err == 0
        _compare(_host(out, f32), exp, f32)


@pytest.mark.parametrize("W,E,K,T,h,pad", [
    (64, 1024, 16, 6, 64, 0.1),    # the library's limits on W, E and top_k
    (4, 8, 4, 33, 32, 0.0),        # top_k > e_local: several experts of a token on one rank
    (1, 6, 3, 50, 64, 0.1),        # one rank: the route is the single fold
    (3, 12, 2, 70, 8, 0.2),        # 16-byte rows, odd sizes
])
def test_agrs_edge_shapes(dev, W, E, K, T, h, pad):
    s = wl.WorkloadSpec("agrs-edge", W=W, E=E, K=K, T=T, h=h, pad_frac=pad, seed=5 * W + E + T)
    x = wl.make(s, num_tokens=np.maximum(T - np.arange(W) % 3, 0).astype(np.int32))
    for f32 in (False, True):
        out, buf = _run(x, dev, f32)
        assert int(buf.status.item()) == 0
        _check_gather(buf, x)
        exp, err = ref.agrs(W, E, K, T, x.a1, x.topk_ids, x.topk_weights, x.num_tokens, f32)
        assert err == 0
        _compare(_host(out, f32), exp, f32)


@pytest.mark.parametrize("cfg", [3, 4, 5])
def test_agrs_full_size_sampled(dev, cfg):
    """Full-size workloads on the GPU against the oracle on sampled tokens: a
    token's output depends on its own row, ids and weights only, so the oracle
    run on the sampled tokens alone (as a smaller batch of the same ranks)
    gives exactly their rows."""
    x = wl.make(cfg)
    s = x.spec
    n = 24
    out, buf = _run(x, dev, out_f32=False)
    assert int(buf.status.item()) == 0
    rng = np.random.default_rng(7 + cfg)
    idx = np.sort(np.stack([rng.choice(s.T, size=n, replace=False) for _ in range(s.W)]), axis=1)
    take = lambda a: np.ascontiguousarray(np.take_along_axis(a, idx[:, :, None], axis=1))
    exp, err = ref.agrs(s.W, s.E, s.K, n, take(x.a1), take(x.topk_ids), take(x.topk_weights))
    assert err == 0
    flat = torch.from_numpy((np.arange(s.W)[:, None] * s.T + idx).reshape(-1)).to(dev)
    got = H.bits_host(out.view(s.W * s.T, s.h).index_select(0, flat))
    _compare(wl.bf16_bits_to_f32(got), exp, False)
    # the gathered copies on the last rank hold every token
    assert torch.equal(buf.x_g[s.W - 1].view(torch.int16),
                       H.bf16_dev(x.a1, dev).view(s.W * s.T, s.h).view(torch.int16))


@pytest.mark.parametrize("cfg,T", [(1, None), (2, None), (4, 64)])
def test_agrs_equals_all_to_all_two_stage_on_gpu(dev, cfg, T):
    """The two routes, both on the GPU: all-to-all dispatch, identity experts
    (expert_out = b_a1) and the two-stage combine give this route's bits."""
    s = wl.spec(cfg, T=T) if T else wl.spec(cfg)
    x = wl.make(s)
    ctx = EpContext(EpConfig(s.W, s.E, s.K, s.T, s.h, sendbuf=True), dev)
    a1, ids, w, nt, _ = H.inputs_dev(x, dev)
    for f32 in (False, True):
        d = ctx.dispatch(a1, ids, w, num_tokens=nt, path="sendbuf")
        two = ctx.combine_two_stage(d.b_a1, out_dtype=torch.float32 if f32 else torch.bfloat16)
        ctx.check()
        out, _ = _run(x, dev, f32)
        assert torch.equal(two.view(torch.int32 if f32 else torch.int16),
                           out.view(torch.int32 if f32 else torch.int16))


def test_agrs_reports_bad_ids_and_counts(dev):
    W, E, K, T, h = 4, 16, 4, 8, 64
    s = wl.WorkloadSpec("agrs-errors", W=W, E=E, K=K, T=T, h=h, seed=11)
    x = wl.make(s)
    x.topk_ids[0, 0] = [3, 99, 3, -1]        # an id >= E and a repeat
    x.topk_ids[2, 5] = [7, 7, 7, 7]          # repeats only
    out, buf = _run(x, dev, out_f32=True)
    code = int(buf.status.item())
    assert code in (L.EP_ERR_EXPERT_ID, L.EP_ERR_DUPLICATE)
    exp, err = ref.agrs(W, E, K, T, x.a1, x.topk_ids, x.topk_weights, x.num_tokens, True)
    assert err & ref.ERR_EXPERT_ID and err & ref.ERR_DUPLICATE
    _compare(_host(out, True), exp, True)
    # a count above max_tokens is reported and clamped, as the oracle does
    x2 = wl.make(s, num_tokens=[T, T + 3, 2, 0])
    out, buf = _run(x2, dev, out_f32=False)
    assert int(buf.status.item()) == L.EP_ERR_CAPACITY
    exp, err = ref.agrs(W, E, K, T, x2.a1, x2.topk_ids, x2.topk_weights, x2.num_tokens, False)
    assert err & ref.ERR_CAPACITY
    _compare(_host(out, False), exp, False)
    # status is cleared by the next clean call
    out, buf = _run(wl.make(s), dev, out_f32=False, buffers=buf)
    assert int(buf.status.item()) == 0


def test_agrs_empty_and_unrouted(dev):
    s = wl.spec(2, T=16)
    x = wl.make(s, num_tokens=[0] * s.W)
    out, _ = _run(x, dev, out_f32=False)
    assert (H.bits_host(out) == 0).all()
    x = wl.make(s)
    x.topk_ids[:] = -1
    out, _ = _run(x, dev, out_f32=True)
    assert (out == 0).all().item()
    # num_tokens omitted: every rank holds max_tokens
    x = wl.make(s)
    out, _ = _run(x, dev, out_f32=False, nt_dev=False)
    exp, _ = ref.agrs(s.W, s.E, s.K, s.T, x.a1, x.topk_ids, x.topk_weights, None, False)
    _compare(_host(out, False), exp, False)


def test_agrs_graph_replay_on_new_inputs(dev):
    s = wl.spec(2, T=32)
    x0, x1 = wl.make(s), wl.make(s, seed=99)
    cfg = _cfg(s)
    a1, ids, w, nt, _ = H.inputs_dev(x0, dev)
    buf = alloc_agrs_buffers(cfg, dev)
    out = torch.empty(s.W, s.T, s.h, dtype=torch.bfloat16, device=dev)
    agrs(cfg, a1, ids, w, num_tokens=nt, buffers=buf, out=out)   # warm-up outside capture
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        agrs(cfg, a1, ids, w, num_tokens=nt, buffers=buf, out=out)
    a1n, idsn, wn, ntn, _ = H.inputs_dev(x1, dev)
    a1.copy_(a1n)
    ids.copy_(idsn)
    w.copy_(wn)
    nt.copy_(ntn)
    g.replay()
    torch.cuda.synchronize(dev)
    exp, _ = ref.agrs(s.W, s.E, s.K, s.T, x1.a1, x1.topk_ids, x1.topk_weights, x1.num_tokens, False)
    _compare(_host(out, False), exp, False)


def test_agrs_worked_example_by_hand(dev):
    """The hand-derived example of tests/golden/agrs_worked_example.json on the
    GPU (its row padded with zeros to the kernels' 8-element granularity): the
    rank-ordered bf16 sums round twice on ties to even and give 1.125 where the
    single fp32 fold gives 1.1328125."""
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "agrs_worked_example.json")))
    W, E, K, Tm, h = g["W"], g["E"], g["top_k"], g["max_tokens"], 8
    a1 = np.zeros((W, Tm, h), np.float32)
    a1[0, 0, :2] = g["a1"]
    ids = np.full((W, Tm, K), -1, np.int32)
    w = np.zeros((W, Tm, K), np.float32)
    ids[0, 0] = g["topk_ids"][0]
    w[0, 0] = g["topk_weights"][0]
    x = wl.Workload(wl.WorkloadSpec("by-hand", W=W, E=E, K=K, T=Tm, h=h), wl.f32_to_bf16_bits(a1), ids, w,
                    np.array(g["num_tokens"], np.int32))
    for f32, key in ((False, "expect_bf16_out"), (True, "expect_f32_out")):
        out, buf = _run(x, dev, f32)
        assert int(buf.status.item()) == 0
        got = _host(out, f32).reshape(W, h)
        assert np.array_equal(got[:, :2], np.array(g[key], np.float32))
        assert (got[:, 2:] == 0).all()
