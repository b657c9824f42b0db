"""Out-of-bounds write detection on the GPU without a sanitizer.

Every output buffer and the workspace are placed inside a larger allocation,
with guard bytes before and after them filled with a fixed pattern. After
dispatch (both paths), combine, the two-stage combine and the all-gather /
reduce-scatter route, the guards must be untouched and the results must still
match the oracle. Bounds checks inside the kernels record errors instead of
trapping, so a bad index shows up here as a changed guard or a status code.
"""
import numpy as np
import pytest
import torch

from combine_ep_route_gb300 import (AgrsBuffers, DispatchOut, EpConfig, EpContext, agrs, workloads as wl)
from combine_ep_route_gb300 import _lib as L
from combine_ep_route_gb300 import ep as E
from oracle import ref
from tests import _gpu_harness as H

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side; a multiple of 256 keeps every buffer's alignment
PATTERN = 0xA5


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


class Guarded:
    """Tensors carved out of guarded byte buffers."""

    def __init__(self, dev):
        self.dev = dev
        self.bufs = []

    def tensor(self, shape, dtype) -> torch.Tensor:
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        buf = torch.full((n + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=self.dev)
        self.bufs.append((buf, n))
        return buf[GUARD:GUARD + n].view(dtype).view(*shape)

    def check(self) -> None:
        torch.cuda.synchronize(self.dev)
        for i, (buf, n) in enumerate(self.bufs):
            head, tail = buf[:GUARD], buf[GUARD + n:]
            assert bool((head == PATTERN).all()), f"buffer {i}: bytes written before its start"
            assert bool((tail == PATTERN).all()), f"buffer {i}: bytes written past its end"


def _dispatch_outputs(g: Guarded, ctx: EpContext, x: wl.Workload) -> DispatchOut:
    s = x.spec
    el = s.E // s.W
    return DispatchOut(
        b_a1=g.tensor((s.W, el, ctx.expert_cap, s.h), torch.bfloat16),
        expert_num_tokens=g.tensor((s.W, el), torch.int32),
        extra_out=[g.tensor((s.W, el, ctx.expert_cap, b), torch.uint8) for b in x.extra_row_bytes])


CASES = [
    (wl.spec(3, T=64), None),
    (wl.spec(4, T=40), None),                                      # an extra payload
    (wl.spec(5, T=12), [12] * 16 + [5] * 8 + [0] * 8),             # ragged, padding rows
    (wl.WorkloadSpec("limits", W=64, E=1024, K=16, T=6, h=64, pad_frac=0.1, seed=9), None),
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("variant", ["fused", "fused_tiled", "sendbuf"])
def test_no_writes_outside_any_buffer(dev, case, variant):
    """These batches are small: "fused" takes the small-batch dispatch,
    "fused_tiled" the tiled one-launch dispatch."""
    s, nt = CASES[case]
    path = "sendbuf" if variant == "sendbuf" else "fused"
    x = wl.make(s, num_tokens=nt)
    g = Guarded(dev)
    cfg = EpConfig(s.W, s.E, s.K, s.T, s.h, extra_row_bytes=tuple(x.extra_row_bytes),
                   sendbuf=path == "sendbuf", zero_pad=True)
    ws = g.tensor((E.workspace_bytes(cfg),), torch.uint8)
    ctx = EpContext(cfg, dev, workspace=ws)
    ctx.set_option(L.EP_OPT_SMALL_DISPATCH, 0 if variant == "fused_tiled" else -1)
    a1, ids, w, ntd, extras = H.inputs_dev(x, dev)
    out = _dispatch_outputs(g, ctx, x)
    ctx.dispatch(a1, ids, w, num_tokens=ntd, extras=extras, out=out, path=path)
    y = g.tensor((s.W, s.T, s.h), torch.bfloat16)
    ctx.combine(out.b_a1, out=y)
    ctx.check()
    g.check()
    m = H.oracle_meta(x)
    H.check_rows(out, m, x, a1, extras)
    exp = ref.combine(m, x.topk_weights, ref.dispatch_rows(m, x.a1))
    assert np.array_equal(H.bits_host(y).reshape(-1, s.h), exp)
    if path == "sendbuf":
        y2 = g.tensor((s.W, s.T, s.h), torch.float32)
        ctx.dispatch(a1, ids, w, num_tokens=ntd, extras=extras, out=out, path=path)
        ctx.combine_two_stage(out.b_a1, out=y2, out_dtype=torch.float32)
        ctx.check()
        g.check()
        assert np.array_equal(y2.cpu().numpy().reshape(-1, s.h),
                              ref.combine_pagemode(m, ref.dispatch_rows(m, x.a1), out_f32=True))


@pytest.mark.parametrize("case", range(len(CASES)))
def test_agrs_no_writes_outside_any_buffer(dev, case):
    s, nt = CASES[case]
    if s.W * s.W * s.T * s.h * 2 > (1 << 30):
        pytest.skip("gathered blocks above 1 GiB")
    x = wl.make(s, num_tokens=nt)
    g = Guarded(dev)
    cfg = EpConfig(s.W, s.E, s.K, s.T, s.h)
    n = s.W * s.T
    buf = AgrsBuffers(x_g=g.tensor((s.W, n, s.h), torch.bfloat16), ids_g=g.tensor((s.W, n, s.K), torch.int32),
                      w_g=g.tensor((s.W, n, s.K), torch.float32), y=g.tensor((s.W, n, s.h), torch.bfloat16),
                      status=g.tensor((1,), torch.int32))
    a1, ids, w, ntd, _ = H.inputs_dev(x, dev)
    y = g.tensor((s.W, s.T, s.h), torch.float32)
    agrs(cfg, a1, ids, w, num_tokens=ntd, out_dtype=torch.float32, buffers=buf, out=y)
    g.check()
    assert int(buf.status.item()) == 0
    exp, err = ref.agrs(s.W, s.E, s.K, s.T, x.a1, x.topk_ids, x.topk_weights, x.num_tokens, True)
    assert err == 0
    assert np.array_equal(y.cpu().numpy().reshape(-1, s.h), exp)
