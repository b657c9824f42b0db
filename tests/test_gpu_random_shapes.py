"""Randomised parity: seeded random problem shapes through the whole path.

Each case draws W, E (a multiple of W), top_k (not always a power of two),
max_tokens (rarely a multiple of the 64-token routing tile), the hidden size,
extra payloads, padding rows, a ragged num_tokens, the dispatch path, whether a
small batch may take the small-batch dispatch, and the output type, then checks
dispatch (metadata and every delivered row, bit for bit) and combine (bit for
bit) against the CPU oracle, and the all-gather / reduce-scatter route on the
same inputs.
"""
import os

import numpy as np
import pytest
import torch

from combine_ep_route_gb300 import agrs, EpConfig, workloads as wl
from combine_ep_route_gb300 import _lib as L
from oracle import ref
from tests import _gpu_harness as H

pytestmark = pytest.mark.gpu

# 300 cases by default (about 6 s); EP_RANDOM_SHAPE_CASES=<n> runs another number (the
# same seeds first; 1000 cases pass in about 20 s)
N_CASES = int(os.environ.get("EP_RANDOM_SHAPE_CASES", "300"))


def _case(i: int):
    rng = np.random.default_rng(20260 + i)
    W = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 16]))
    e_local = int(rng.choice([1, 2, 3, 4, 6, 8, 16]))
    E = W * e_local
    K = int(rng.integers(1, min(E, 16) + 1))
    T = int(rng.integers(1, 200))
    h = int(8 * rng.integers(1, 65))
    pad = float(rng.choice([0.0, 0.1, 0.3]))
    extras = tuple(int(c) for c in rng.choice([4, 8, 16], size=int(rng.integers(0, 3))))
    spec = wl.WorkloadSpec(f"random-{i}", W=W, E=E, K=K, T=T, h=h, pad_frac=pad,
                           extra_f32_cols=extras, seed=int(rng.integers(1 << 30)))
    nt = None
    if rng.random() < 0.5:
        nt = rng.integers(0, T + 1, size=W).astype(np.int32)
    path = "sendbuf" if rng.random() < 0.4 else "fused"
    out_f32 = bool(rng.random() < 0.3)
    small = -1 if rng.random() < 0.5 else 0   # small-batch dispatch allowed, or the tiled one
    return spec, nt, path, out_f32, small


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape(dev, i):
    spec, nt, path, out_f32, small = _case(i)
    x = wl.make(spec, num_tokens=nt)
    s = x.spec
    ctx = H.make_ctx(x, dev, sendbuf=path == "sendbuf")
    ctx.set_option(L.EP_OPT_SMALL_DISPATCH, small)
    a1, ids, w, ntd, extras = H.inputs_dev(x, dev)
    out = ctx.dispatch(a1, ids, w, num_tokens=ntd, extras=extras, path=path)
    ctx.check()
    m = H.oracle_meta(x)
    assert m.err == 0
    H.check_meta(ctx, m, x, out.expert_num_tokens)
    H.check_rows(out, m, x, a1, extras)
    packed = H.fill_pool_rows(out, m, s.h, i)
    H.check_combine(ctx, out.b_a1, m, x, packed, out_f32)
    # the other route on the same tokens
    if s.W * s.W * s.T * s.h * 2 <= (256 << 20):
        y = agrs(EpConfig(s.W, s.E, s.K, s.T, s.h), a1, ids, w, num_tokens=ntd,
                 out_dtype=torch.float32 if out_f32 else torch.bfloat16)
        torch.cuda.synchronize(dev)
        exp, err = ref.agrs(s.W, s.E, s.K, s.T, x.a1, x.topk_ids, x.topk_weights, x.num_tokens, out_f32)
        assert err == 0
        got = y.cpu().numpy() if out_f32 else H.bits_host(y)
        assert np.array_equal(got.reshape(exp.shape), exp)
