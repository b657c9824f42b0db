"""ep_route_static: routing for callers that cannot allocate device memory.

Some callers cannot use ep_ctx_create's workspace because they may not
allocate: an inference engine that owns and plans all device memory at
start-up, a plugin whose host framework forbids allocation after
initialisation, or a latency-critical path where a cudaMalloc could
synchronise the device. ep_route_static serves them with its scratch in a
fixed static device array. This file checks, through the C-ABI, that two
calls in a row give exactly the routing metadata ep_dispatch produces for the
same inputs (all integer or copied values, so bit-exact), and that a problem
larger than the fixed scratch is refused. It is collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from combine_ep_route_gb300 import _lib as L, workloads as wl
from tests import _gpu_harness as H

KEYS = ("send_cnt", "pair_row", "pair_w", "pair_send", "recv_eloc", "recv_w", "recv_row")


def _cfg(s):
    c = L.EpConfigC()
    c.W, c.E, c.top_k, c.max_tokens, c.hidden, c.x_dtype = s.W, s.E, s.K, s.T, s.h, L.EP_BF16
    return c


def _existing(x, dev, expect_status=0):
    """Routing metadata through the existing entry point (ep_dispatch), and the
    device-side status ep_status reports for it."""
    ctx = H.make_ctx(x, dev)
    a1, ids, w, nt, extras = H.inputs_dev(x, dev)
    out = ctx.dispatch(a1, ids, w, num_tokens=nt, extras=extras)
    assert ctx.status() == expect_status
    got = {k: v.clone() for k, v in ctx.metadata().items() if k in KEYS}
    got["expert_num_tokens"] = out.expert_num_tokens.clone()
    ctx.reset()
    return got


def _static_call(x, dev):
    """One ep_route_static call; the test owns every buffer (the entry point allocates nothing)."""
    s = x.spec
    S = min(s.K, s.E // s.W)
    i32, f32 = torch.int32, torch.float32
    bufs = {
        "send_cnt": torch.full((s.W, s.W), -7, dtype=i32, device=dev),
        "pair_row": torch.full((s.W, s.T, s.K), -7, dtype=i32, device=dev),
        "pair_w": torch.full((s.W, s.T, s.K), -7.0, dtype=f32, device=dev),
        "pair_send": torch.full((s.W, s.T, s.K), -7, dtype=i32, device=dev),
        "recv_eloc": torch.full((s.W, s.W, s.T, S), -7, dtype=i32, device=dev),
        "recv_w": torch.full((s.W, s.W, s.T, S), -7.0, dtype=f32, device=dev),
        "recv_row": torch.full((s.W, s.W, s.T, S), -7, dtype=i32, device=dev),
        "expert_num_tokens": torch.full((s.W, s.E // s.W), -7, dtype=i32, device=dev),
    }
    status = torch.full((1,), 12345, dtype=i32, device=dev)
    o = L.EpRouteOutputsC()
    for k, v in bufs.items():
        setattr(o, k, v.data_ptr())
    o.status = status.data_ptr()
    _, ids, w, nt, _ = H.inputs_dev(x, dev)
    rc = L.lib().ep_route_static(C.byref(_cfg(s)), nt.data_ptr(), ids.data_ptr(), w.data_ptr(),
                                 C.byref(o), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, L.lib().ep_error_string(rc)
    return bufs, status, (ids, w, nt)


def _same(x, exp, got):
    s = x.spec
    cnt = exp["send_cnt"].cpu().numpy()
    valid = np.arange(s.T)[None, None, :] < cnt.T[:, :, None]   # received slots [d][s][slot]
    for k in KEYS + ("expert_num_tokens",):
        e, g = exp[k].cpu().numpy(), got[k].cpu().numpy()
        if k.startswith("recv_"):
            e, g = e[valid], g[valid]
        assert np.array_equal(e.view(np.uint32), g.view(np.uint32)), k


@pytest.mark.gpu
def test_static_routing_matches_dispatch_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    xa = wl.make(3)                          # prefill shape: 8 ranks x 1024 tokens, E=256
    xb = wl.make(wl.spec(5, T=128))          # another shape and id mix, with padding rows
    exp_a, exp_b = _existing(xa, dev), _existing(xb, dev)
    got_a, st_a, keep_a = _static_call(xa, dev)
    got_b, st_b, keep_b = _static_call(xb, dev)  # second call in a row reuses the array
    torch.cuda.synchronize()
    assert int(st_a.item()) == 0 and int(st_b.item()) == 0
    _same(xa, exp_a, got_a)
    _same(xb, exp_b, got_b)
    # a third call: a ragged batch with one id repeated inside a token row; the
    # status word must carry the code ep_status reports for the same inputs
    xc = wl.make(wl.spec(2, T=96), num_tokens=np.array([96, 0, 17, 64, 95, 1, 50, 96], np.int32))
    t = int(np.nonzero((xc.topk_ids[2, :17] >= 0).all(axis=1))[0][0])   # a routed token of rank 2
    xc.topk_ids[2, t, 3] = xc.topk_ids[2, t, 1]
    exp_c = _existing(xc, dev, expect_status=L.EP_ERR_DUPLICATE)
    got_c, st_c, keep_c = _static_call(xc, dev)
    torch.cuda.synchronize()
    assert int(st_c.item()) == L.EP_ERR_DUPLICATE
    _same(xc, exp_c, got_c)


def test_static_routing_refuses_misaligned_pointers():
    """Host-side check, no GPU work: one pointer off a 4-byte boundary at a time
    is refused with EP_ERR_INVALID_ARG before anything is enqueued."""
    from combine_ep_route_gb300 import build
    build.build()
    c = L.EpConfigC()
    c.W, c.E, c.top_k, c.max_tokens, c.hidden, c.x_dtype = 2, 8, 2, 16, 64, L.EP_BF16
    base = 0x7F0000000000
    names = [f for f, _ in L.EpRouteOutputsC._fields_]
    for bad in names + ["num_tokens", "topk_ids", "topk_weights"]:
        o = L.EpRouteOutputsC()
        for i, f in enumerate(names):
            setattr(o, f, base + 0x100000 * (i + 1) + (2 if f == bad else 0))
        nt = base + (2 if bad == "num_tokens" else 0)
        ids = base + 0x40000000 + (2 if bad == "topk_ids" else 0)
        w = base + 0x50000000 + (2 if bad == "topk_weights" else 0)
        rc = L.lib().ep_route_static(C.byref(c), nt, ids, w, C.byref(o), None)
        assert rc == L.EP_ERR_INVALID_ARG, bad


def test_static_routing_refuses_problems_beyond_its_scratch():
    from combine_ep_route_gb300 import build
    build.build()
    c = L.EpConfigC()
    c.W, c.E, c.top_k, c.max_tokens, c.hidden, c.x_dtype = 64, 1024, 8, 8192, 128, L.EP_BF16
    o = L.EpRouteOutputsC()
    for f, _ in o._fields_:
        setattr(o, f, 0x7F0000000000)
    rc = L.lib().ep_route_static(C.byref(c), None, o.pair_row, o.pair_w, C.byref(o), None)
    assert rc == L.EP_ERR_SCRATCH_LIMIT
    assert "static scratch" in L.lib().ep_error_string(rc).decode()
