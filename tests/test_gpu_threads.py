"""Two host threads, each with its own context and stream, dispatching and
combining at the same time on one GPU: the launch helpers' shared-memory limit
table (one record per kernel and device, under a lock) is used from both
threads, and every result must still match the oracle."""
import threading

import numpy as np
import pytest
import torch

from combine_ep_route_gb300 import workloads as wl
from tests import _gpu_harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def _worker(x, dev, reps, errors):
    try:
        torch.cuda.set_device(dev)
        s = x.spec
        stream = torch.cuda.Stream(dev)
        ctx = H.make_ctx(x, dev)
        with torch.cuda.stream(stream):
            a1, ids, w, nt, extras = H.inputs_dev(x, dev)
            out = ctx.alloc_dispatch_outputs()
            y = torch.empty((s.W, s.T, s.h), dtype=torch.bfloat16, device=dev)
            for _ in range(reps):
                ctx.dispatch(a1, ids, w, num_tokens=nt, extras=extras, out=out, stream=stream)
                ctx.combine(out.b_a1, out=y, stream=stream)
        ctx.check(stream)
        m = H.oracle_meta(x)
        H.check_meta(ctx, m, x, out.expert_num_tokens)
        H.check_rows(out, m, x, a1, extras)
        routed = (x.topk_ids >= 0).any(axis=2)
        got = H.bits_host(y).reshape(s.W, s.T, s.h)
        assert np.array_equal(got[routed], x.a1[routed])      # identity experts, weights sum to 1
    except BaseException as e:   # reported by the main thread
        errors.append(e)


def test_two_host_threads_two_contexts(dev):
    # shapes that take different kernels and shared-memory sizes: the tiled
    # one-launch dispatch (prefill rows) and the small-batch one (decode)
    xs = [wl.make(wl.spec(3, T=256)), wl.make(2)]
    errors = []
    threads = [threading.Thread(target=_worker, args=(x, dev, 10, errors)) for x in xs]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads), "a worker did not finish"
    if errors:
        raise errors[0]
