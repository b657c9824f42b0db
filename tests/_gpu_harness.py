"""Helpers of the GPU parity tests: run the CUDA path through the binding and
compare what it produced with the CPU oracle (dispatch bit-exact, combine
within the stated tolerance and, by construction of the fold, bit-exact)."""
from __future__ import annotations

import numpy as np
import torch

from combine_ep_route_gb300 import EpConfig, EpContext, workloads as wl
from oracle import ref
from tests._metrics import max_rel_err, TOL_BF16_OUT, TOL_F32_OUT


def bf16_dev(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def bits_host(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def make_ctx(x: wl.Workload, dev, **kw) -> EpContext:
    s = x.spec
    cfg = EpConfig(s.W, s.E, s.K, s.T, s.h, extra_row_bytes=tuple(x.extra_row_bytes), **kw)
    return EpContext(cfg, dev)


def inputs_dev(x: wl.Workload, dev):
    a1 = bf16_dev(x.a1, dev)
    ids = torch.from_numpy(x.topk_ids).to(dev)
    w = torch.from_numpy(x.topk_weights).to(dev)
    nt = torch.from_numpy(x.num_tokens).to(dev)
    extras = [torch.from_numpy(e).to(dev) for e in x.extras]
    return a1, ids, w, nt, extras


def oracle_meta(x: wl.Workload) -> ref.Meta:
    s = x.spec
    return ref.dispatch_meta(s.W, s.E, s.K, s.T, x.topk_ids, x.topk_weights, x.num_tokens)


def expected_recv_row(m: ref.Meta) -> np.ndarray:
    out = np.full((m.W, m.W, m.Tm, m.S), -1, np.int32)
    e, row = np.nonzero(m.row_src >= 0)
    src = m.row_src[e, row]
    out[e // m.e_local, src // m.Tm, src % m.Tm, m.row_col[e, row]] = row
    return out


def expected_pair_send(m: ref.Meta) -> np.ndarray:
    out = np.full((m.W, m.Tm, m.K), -1, np.int32)
    s, d, q = np.nonzero(m.send_tok >= 0)
    t = m.send_tok[s, d, q]
    k = m.send_k[s, d, q, 0]
    out[s, t, k] = (s * m.W + d) * m.Tm + q
    return out


def check_meta(ctx: EpContext, m: ref.Meta, x: wl.Workload, ent: torch.Tensor) -> None:
    md = {k: v.cpu().numpy() for k, v in ctx.metadata().items() if k not in ("send_x", "recv_x")}
    assert np.array_equal(ent.cpu().numpy(), m.expert_num_tokens), "expert_num_tokens"
    assert np.array_equal(md["send_cnt"], m.send_cnt), "send_cnt"
    assert np.array_equal(md["pair_row"], m.pair_row), "pair_row (combine map / slot order)"
    want_w = np.where(m.pair_row >= 0, x.topk_weights, np.float32(0))
    assert np.array_equal(md["pair_w"], want_w), "pair_w"
    assert np.array_equal(md["pair_send"], expected_pair_send(m)), "pair_send"
    valid = np.arange(m.Tm)[None, None, :] < m.recv_cnt[:, :, None]
    assert np.array_equal(md["recv_eloc"][valid], m.recv_eloc[valid]), "recv_eloc"
    assert np.array_equal(md["recv_w"][valid], m.recv_w[valid]), "recv_w"
    assert np.array_equal(md["recv_row"][valid], expected_recv_row(m)[valid]), "recv_row"


def valid_rows(m: ref.Meta):
    """Flat (e*Ecap+row) index and source token of every delivered row, in (e, row) order."""
    rt = m.row_token()
    e, row = np.nonzero(rt >= 0)
    return e.astype(np.int64) * m.Ecap + row, rt[e, row]


def check_rows(out, m: ref.Meta, x: wl.Workload, a1: torch.Tensor, extras) -> None:
    s = x.spec
    flat, tok = valid_rows(m)
    dev = a1.device
    fi = torch.from_numpy(flat).to(dev)
    ti = torch.from_numpy(tok).to(dev)
    got = out.b_a1.view(-1, s.h).view(torch.int16).index_select(0, fi)
    exp = a1.view(-1, s.h).view(torch.int16).index_select(0, ti)
    assert torch.equal(got, exp), "b_a1 rows differ from the source tokens the oracle names"
    for i, (xo, xi) in enumerate(zip(out.extra_out, extras)):
        nb = x.extra_row_bytes[i]
        g2 = xo.view(-1, nb).index_select(0, fi)
        e2 = xi.view(-1, nb).index_select(0, ti)
        assert torch.equal(g2, e2), f"extra payload {i} rows differ"


def fill_pool_rows(out, m: ref.Meta, h: int, seed: int):
    """Overwrite the delivered rows of b_a1 with rows drawn from a seeded pool
    (the expert outputs of the combine test); return them packed for the oracle."""
    rng = np.random.default_rng(seed)
    P = 1021
    pool = wl.f32_to_bf16_bits(rng.standard_normal((P, h), dtype=np.float32))
    flat, _ = valid_rows(m)
    idx = (flat * 2654435761) % P
    packed = pool[idx]
    dev = out.b_a1.device
    b = out.b_a1.view(-1, h)
    b.index_copy_(0, torch.from_numpy(flat).to(dev), bf16_dev(pool, dev).index_select(
        0, torch.from_numpy(idx).to(dev)))
    return packed


def check_combine(ctx: EpContext, expert_out: torch.Tensor, m: ref.Meta, x: wl.Workload,
                  packed: np.ndarray, out_f32: bool) -> None:
    s = x.spec
    dt = torch.float32 if out_f32 else torch.bfloat16
    got = ctx.combine(expert_out, out_dtype=dt)
    ctx.check()
    exp = ref.combine(m, x.topk_weights, packed, out_f32=out_f32)
    if out_f32:
        g = got.cpu().numpy().reshape(-1, s.h)
        e = exp
        tol = TOL_F32_OUT
    else:
        g = wl.bf16_bits_to_f32(bits_host(got).reshape(-1, s.h))
        e = wl.bf16_bits_to_f32(exp)
        tol = TOL_BF16_OUT
    # rows of tokens that do not exist (t >= num_tokens) and padding rows are zero
    err = max_rel_err(g, e)
    assert err <= tol, f"combine max relative error {err} > {tol}"
    # the kernel folds in the same order with the same roundings: identical bits
    assert np.array_equal(g.view(np.uint32), e.view(np.uint32)), "combine not bit-identical to the oracle"
