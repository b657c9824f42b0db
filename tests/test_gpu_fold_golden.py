"""GPU: the hand-derived rounding golden (tests/golden/fold_rounding.json) through
the C-ABI.

The page's finalize rounds each weighted row to fp32 before it accumulates it,
so a kernel that fused a product into its sum (an FMA) would give 2^-30 or
-2^-23 where the golden says +0, and one fp32 ulp more on a positive-weight tie;
a kernel that folded the top-k pairs in another order would give 1 + 2^-23
where the golden says 1. Checked on both dispatch paths with identity experts,
on the single-fold combine (bf16 and fp32 out), the two-stage combine and the
all-gather / reduce-scatter route, bit for bit.
"""
import json
import os

import numpy as np
import pytest
import torch

from combine_ep_route_gb300 import EpConfig, EpContext, agrs, alloc_agrs_buffers, workloads as wl
from tests import _gpu_harness as H

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fold_rounding.json")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


@pytest.fixture(scope="module")
def golden():
    g = json.load(open(GOLDEN))
    a1f = np.array(g["a1"], np.float32)
    return dict(W=g["W"], E=g["E"], K=g["K"], Tm=g["Tm"], h=g["h"],
                ids=np.array(g["topk_ids"], np.int32),
                w=np.array(g["topk_weights"], np.float32),
                a1=wl.f32_to_bf16_bits(a1f),
                nt=np.array(g["num_tokens"], np.int32),
                expect=np.array(g["expect_out"], np.float32))


def _host(y: torch.Tensor) -> np.ndarray:
    if y.dtype == torch.float32:
        return y.cpu().numpy()
    return wl.bf16_bits_to_f32(H.bits_host(y))


def _same_bits(got: np.ndarray, expect: np.ndarray) -> bool:
    got = got.reshape(expect.shape).astype(np.float32)
    return np.array_equal(got.view(np.uint32), expect.view(np.uint32))


@pytest.mark.parametrize("path", ["fused", "sendbuf"])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_combines_match_the_hand_derived_rounding(dev, golden, path, out_dtype):
    g = golden
    cfg = EpConfig(g["W"], g["E"], g["K"], g["Tm"], g["h"], sendbuf=(path == "sendbuf"))
    ctx = EpContext(cfg, dev)
    a1 = H.bf16_dev(g["a1"], dev)
    ids = torch.from_numpy(g["ids"]).to(dev)
    w = torch.from_numpy(g["w"]).to(dev)
    nt = torch.from_numpy(g["nt"]).to(dev)
    out = ctx.dispatch(a1, ids, w, num_tokens=nt, path=path)
    y = ctx.combine(out.b_a1, out_dtype=out_dtype)        # identity experts
    ctx.check()
    assert _same_bits(_host(y), g["expect"]), _host(y)
    if path == "sendbuf":
        ctx.dispatch(a1, ids, w, num_tokens=nt, out=out, path=path)
        y2 = ctx.combine_two_stage(out.b_a1, out_dtype=out_dtype)
        ctx.check()
        assert _same_bits(_host(y2), g["expect"]), _host(y2)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_agrs_route_matches_the_hand_derived_rounding(dev, golden, out_dtype):
    g = golden
    cfg = EpConfig(g["W"], g["E"], g["K"], g["Tm"], g["h"])
    a1 = H.bf16_dev(g["a1"], dev)
    ids = torch.from_numpy(g["ids"]).to(dev)
    w = torch.from_numpy(g["w"]).to(dev)
    nt = torch.from_numpy(g["nt"]).to(dev)
    buf = alloc_agrs_buffers(cfg, dev)
    y = agrs(cfg, a1, ids, w, num_tokens=nt, out_dtype=out_dtype, buffers=buf)
    torch.cuda.synchronize(dev)
    assert int(buf.status.item()) == 0
    assert _same_bits(_host(y), g["expect"]), _host(y)
