"""Python face of the C oracle (``ep_oracle.c``): routed MoE EP dispatch / combine.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg are the only callers. Nothing here touches the CUDA library.

The functions restate vLLM ``AllToAllBatchedPrepareAndFinalize`` (page
fused_moe/prepare_finalize/alltoall_batched): ``capacities``, ``prepare``
(route, pack, all_to_all_single, deliver) and ``finalize`` (weighted reduce,
all_to_all_single back, per-token sum). See ``ep_oracle.c`` for the readings
taken where the page is open.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass
from typing import Optional

import numpy as np

from . import build as _build

ERR_EXPERT_ID = 1
ERR_DUPLICATE = 2
ERR_CAPACITY = 4

_lib = None
_openmp = False


def use_openmp(on: bool = True) -> None:
    """Load the -fopenmp build of the same oracle source from the next call on
    (for timing on all host cores; results are identical). Call it before the
    first oracle call of the process."""
    global _lib, _openmp
    _openmp = bool(on)
    _lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(_build.build(openmp=_openmp))
        P = C.c_void_p
        i = C.c_int
        _lib.oracle_capacities.argtypes = [i, i, i, i, P, P, P]
        _lib.oracle_route.argtypes = [i, i, i, i, P, P, P, P, P, P, P, P, P]
        _lib.oracle_exchange_meta.argtypes = [i, i, i, i, P, P, P, P, P, P]
        _lib.oracle_deliver_meta.argtypes = [i, i, i, i, P, P, P, P, P, P]
        _lib.oracle_pair_rows.argtypes = [i, i, i, i, P, P, P, P, P, P]
        _lib.oracle_pack.argtypes = [i, i, C.c_size_t, P, P, P, P]
        _lib.oracle_exchange.argtypes = [i, i, C.c_size_t, P, P]
        _lib.oracle_deliver.argtypes = [i, i, i, C.c_size_t, P, P, P, P, P]
        _lib.oracle_combine.argtypes = [i, i, i, i, i, P, P, P, P, P, i, P, P, C.c_int64]
        _lib.oracle_combine_pagemode.argtypes = [i, i, i, i, i, P, P, P, P, P, P, P, i, P]
        _lib.oracle_scale_input.argtypes = [C.c_int64, i, P, P, P]
        _lib.oracle_agrs.argtypes = [i, i, i, i, i, P, P, P, P, i, P, P]
        for f in ("oracle_capacities", "oracle_route", "oracle_exchange_meta",
                  "oracle_deliver_meta", "oracle_pair_rows", "oracle_pack", "oracle_exchange",
                  "oracle_deliver", "oracle_combine", "oracle_combine_pagemode",
                  "oracle_scale_input", "oracle_agrs"):
            getattr(_lib, f).restype = None
    return _lib


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def capacities(W: int, E: int, K: int, Tm: int):
    """``capacities(topk)``: (token slots per rank, expert slots per token, rows per expert)."""
    a, b, c = C.c_int(), C.c_int(), C.c_int()
    lib().oracle_capacities(W, E, K, Tm, C.byref(a), C.byref(b), C.byref(c))
    return a.value, b.value, c.value


@dataclass
class Meta:
    """Dispatch metadata of all W ranks (every array C-contiguous)."""
    W: int
    E: int
    K: int
    Tm: int
    S: int
    Ecap: int
    num_tokens: np.ndarray         # [W]
    send_cnt: np.ndarray           # [W(s), W(d)]
    send_tok: np.ndarray           # [W(s), W(d), Tm]
    send_eloc: np.ndarray          # [W(s), W(d), Tm, S]
    send_w: np.ndarray             # [W(s), W(d), Tm, S]
    send_k: np.ndarray             # [W(s), W(d), Tm, S]
    recv_cnt: np.ndarray           # [W(d), W(s)]
    recv_eloc: np.ndarray          # [W(d), W(s), Tm, S]
    recv_w: np.ndarray             # [W(d), W(s), Tm, S]
    expert_num_tokens: np.ndarray  # [W(d), e_local]
    row_src: np.ndarray            # [E, Ecap]  s*Tm+slot, -1
    row_col: np.ndarray            # [E, Ecap]
    pair_row: np.ndarray           # [W, Tm, K] flat (d*e_local+j)*Ecap+row, -1
    row_off: np.ndarray            # [E] int64: start of expert e in packed row tables
    err: int

    @property
    def e_local(self) -> int:
        return self.E // self.W

    @property
    def n_rows(self) -> int:
        return int(self.expert_num_tokens.sum())

    def row_token(self) -> np.ndarray:
        """[E, Ecap] flat source token (s*Tm+t) held by each delivered row, -1 past the count."""
        out = np.full(self.row_src.shape, -1, dtype=np.int64)
        m = self.row_src >= 0
        s = self.row_src[m] // self.Tm
        slot = self.row_src[m] % self.Tm
        d = np.nonzero(m)[0] // self.e_local
        t = self.send_tok[s, d, slot]
        out[m] = s * self.Tm + t
        return out


def dispatch_meta(W: int, E: int, K: int, Tm: int, topk_ids: np.ndarray,
                  topk_weights: np.ndarray, num_tokens: Optional[np.ndarray] = None) -> Meta:
    """Routing, slots, exchange of the metadata and delivery rows (no payload bytes)."""
    L = lib()
    _, S, Ecap = capacities(W, E, K, Tm)
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32).reshape(W, Tm, K)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32).reshape(W, Tm, K)
    nt = (np.full(W, Tm, dtype=np.int32) if num_tokens is None
          else np.ascontiguousarray(num_tokens, dtype=np.int32).reshape(W))
    err = C.c_uint32(0)
    send_cnt = np.empty((W, W), np.int32)
    send_tok = np.empty((W, W, Tm), np.int32)
    send_eloc = np.empty((W, W, Tm, S), np.int32)
    send_w = np.empty((W, W, Tm, S), np.float32)
    send_k = np.empty((W, W, Tm, S), np.int32)
    L.oracle_route(W, E, K, Tm, _p(nt), _p(ids), _p(w), _p(send_cnt), _p(send_tok),
                   _p(send_eloc), _p(send_w), _p(send_k), C.byref(err))
    recv_cnt = np.empty((W, W), np.int32)
    recv_eloc = np.empty_like(send_eloc)
    recv_w = np.empty_like(send_w)
    L.oracle_exchange_meta(W, E, K, Tm, _p(send_cnt), _p(send_eloc), _p(send_w), _p(recv_cnt),
                           _p(recv_eloc), _p(recv_w))
    e_local = E // W
    ent = np.empty((W, e_local), np.int32)
    row_src = np.empty((E, Ecap), np.int32)
    row_col = np.empty((E, Ecap), np.int32)
    L.oracle_deliver_meta(W, E, K, Tm, _p(recv_cnt), _p(recv_eloc), _p(ent), _p(row_src),
                          _p(row_col), C.byref(err))
    pair_row = np.empty((W, Tm, K), np.int32)
    L.oracle_pair_rows(W, E, K, Tm, _p(ent), _p(row_src), _p(row_col), _p(send_tok), _p(send_k),
                       _p(pair_row))
    cnt = ent.reshape(-1).astype(np.int64)
    row_off = np.zeros(E, np.int64)
    row_off[1:] = np.cumsum(cnt)[:-1]
    return Meta(W, E, K, Tm, S, Ecap, nt, send_cnt, send_tok, send_eloc, send_w, send_k,
                recv_cnt, recv_eloc, recv_w, ent, row_src, row_col, pair_row, row_off,
                int(err.value))


def dispatch_rows(meta: Meta, rows: np.ndarray) -> np.ndarray:
    """Payload of the dispatch: pack, exchange, deliver.

    ``rows`` is ``[W, Tm, rb]`` bytes per token (an activation row, possibly
    followed by extra payload bytes). Returns the delivered rows packed in (d,
    j, row) order, ``[n_rows, rb]``; expert e starts at ``meta.row_off[e]``.
    """
    L = lib()
    W, Tm = meta.W, meta.Tm
    src = np.ascontiguousarray(rows).view(np.uint8).reshape(W, Tm, -1)
    rb = src.shape[2]
    send_x = np.empty((W, W, Tm, rb), np.uint8)
    L.oracle_pack(W, Tm, rb, _p(meta.send_cnt), _p(meta.send_tok), _p(src), _p(send_x))
    recv_x = np.empty_like(send_x)
    L.oracle_exchange(W, Tm, rb, _p(send_x), _p(recv_x))
    del send_x
    out = np.empty((meta.n_rows, rb), np.uint8)
    L.oracle_deliver(W, meta.E, Tm, rb, _p(meta.expert_num_tokens), _p(meta.row_src),
                     _p(recv_x), _p(meta.row_off), _p(out))
    return out


def _rows2d(meta: Meta, expert_rows: np.ndarray) -> np.ndarray:
    """Packed rows as a C-contiguous [n_rows, h] uint16 array (h read from the
    array's last axis, so an empty table keeps its width)."""
    x = np.ascontiguousarray(expert_rows).view(np.uint16)
    if x.ndim != 2:
        x = x.reshape(meta.n_rows, -1)
    assert x.shape[0] == meta.n_rows
    return x


def combine(meta: Meta, topk_weights: np.ndarray, expert_rows: np.ndarray, out_f32: bool = False,
            tokens: Optional[np.ndarray] = None) -> np.ndarray:
    """``finalize`` with the fixed top-k-order fp32 fold, rounded once.

    ``expert_rows``: packed expert-output rows ``[n_rows, h]`` as bf16 bits
    (uint16), in the (d, j, row) order of :func:`dispatch_rows`. Returns
    ``[W*Tm, h]`` (bf16 bits or float32); with ``tokens`` only those flat token
    rows are computed (the others are left zero).
    """
    L = lib()
    W, Tm, K = meta.W, meta.Tm, meta.K
    x = _rows2d(meta, expert_rows)
    h = x.shape[1]
    w = np.ascontiguousarray(topk_weights, dtype=np.float32).reshape(W, Tm, K)
    out = np.zeros((W * Tm, h), np.float32 if out_f32 else np.uint16)
    tk = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int64)
    L.oracle_combine(W, meta.E, K, Tm, h, _p(meta.num_tokens), _p(meta.pair_row), _p(w), _p(x),
                     _p(meta.row_off), int(out_f32), _p(out), _p(tk),
                     0 if tk is None else len(tk))
    return out


def combine_pagemode(meta: Meta, expert_rows: np.ndarray, out_f32: bool = False) -> np.ndarray:
    """``finalize`` in the page's two-stage rounding (see ``oracle_combine_pagemode``)."""
    L = lib()
    W, Tm, K, S = meta.W, meta.Tm, meta.K, meta.S
    x = _rows2d(meta, expert_rows)
    h = x.shape[1]
    # flat row of each column of each send slot
    rs = np.full((W, W, Tm, S), -1, np.int32)
    s_idx, d_idx, q_idx, c_idx = np.nonzero(meta.send_k >= 0)
    t = meta.send_tok[s_idx, d_idx, q_idx]
    k = meta.send_k[s_idx, d_idx, q_idx, c_idx]
    rs[s_idx, d_idx, q_idx, c_idx] = meta.pair_row[s_idx, t, k]
    out = np.zeros((W * Tm, h), np.float32 if out_f32 else np.uint16)
    L.oracle_combine_pagemode(W, meta.E, K, Tm, h, _p(meta.send_cnt), _p(meta.send_tok),
                              _p(meta.send_eloc), _p(meta.send_w), _p(rs), _p(x),
                              _p(meta.row_off), int(out_f32), _p(out))
    return out


def scale_input(a1: np.ndarray, topk_weights: np.ndarray) -> np.ndarray:
    """``prepare``'s apply_router_weight_on_input (top_k == 1): a1 * bf16(w) rounded
    to bf16, per token. a1: [..., h] bf16 bits; topk_weights: [..., 1]."""
    x = np.ascontiguousarray(a1).view(np.uint16)
    h = x.shape[-1]
    n = x.size // h
    w = np.ascontiguousarray(topk_weights, dtype=np.float32).reshape(-1)
    assert w.size == n, "apply_router_weight_on_input needs top_k == 1"
    out = np.empty_like(x)
    lib().oracle_scale_input(n, h, _p(x), _p(w), _p(out))
    return out


def agrs(W: int, E: int, K: int, Tm: int, a1: np.ndarray, topk_ids: np.ndarray,
         topk_weights: np.ndarray, num_tokens: Optional[np.ndarray] = None,
         out_f32: bool = False):
    """The all-gather / reduce-scatter route with identity experts (see
    ``oracle_agrs``). Returns (out [W*Tm, h], error bits)."""
    x = np.ascontiguousarray(a1).view(np.uint16).reshape(W * Tm, -1)
    h = x.shape[1]
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32).reshape(W, Tm, K)
    w = np.ascontiguousarray(topk_weights, dtype=np.float32).reshape(W, Tm, K)
    nt = (np.full(W, Tm, dtype=np.int32) if num_tokens is None
          else np.ascontiguousarray(num_tokens, dtype=np.int32).reshape(W))
    out = np.zeros((W * Tm, h), np.float32 if out_f32 else np.uint16)
    err = C.c_uint32(0)
    lib().oracle_agrs(W, E, K, Tm, h, _p(nt), _p(ids), _p(w), _p(x), int(out_f32), _p(out),
                      C.byref(err))
    return out, int(err.value)
