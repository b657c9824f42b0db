"""Seeded synthetic inputs for routed MoE expert-parallel dispatch / combine.

This module only draws random inputs. It holds none of the routing, slot or
combine arithmetic, so both the CPU oracle (under ``oracle/``) and the CUDA
path may take their inputs from it.

Every workload simulates ``W`` expert-parallel ranks; every array carries a
leading ``[W]`` rank dimension:

* ``a1``          ``[W, T, h]``  bf16 bit patterns (``uint16``), N(0,1) rounded
                                 to nearest-even;
* ``topk_ids``    ``[W, T, K]``  int32 expert ids, ``-1`` on padding rows;
* ``topk_weights````[W, T, K]``  float32, softmax over K of N(0,1) logits;
* ``num_tokens``  ``[W]``        int32, tokens held by each rank (``T`` unless
                                 a ragged batch is asked for);
* ``extras``      list of ``[W, T, bytes]`` uint8 opaque payload rows.

The five named workloads follow the batch shapes of the routed all-to-all
batched prepare/finalize page (vLLM ``AllToAllBatchedPrepareAndFinalize``,
``prepare``): a decode-size batch, a prefill-size batch, a skewed-popularity
batch with a second payload (the multi-payload dispatch of FlashInfer's
``MoeAlltoAll.dispatch``), and a wide batch with rank-local expert groups.
Draw order inside one workload is fixed: a1, expert ids, padding rows, weight
logits, extra payloads.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np

__all__ = ["WorkloadSpec", "Workload", "SPECS", "make", "spec", "f32_to_bf16_bits",
           "bf16_bits_to_f32"]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the bit patterns."""
    u = np.array(x, dtype=np.float32, copy=True).view(np.uint32)
    if not np.isfinite(x).all():
        raise ValueError("only finite values are drawn")
    lsb = u >> 16
    lsb &= 1
    u += np.uint32(0x7FFF)   # finite |x| < 2^127: no wrap-around
    u += lsb
    u >>= 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass(frozen=True)
class WorkloadSpec:
    name: str
    W: int                 # simulated expert-parallel ranks
    E: int                 # experts in total (E % W == 0)
    K: int                 # top_k
    T: int                 # tokens per rank (= max_tokens)
    h: int                 # hidden size (bf16 elements per a1 row)
    ids: str = "uniform"   # "uniform" | "zipf" | "grouped"
    pad_frac: float = 0.0  # share of rows per rank whose ids are all -1
    zipf_s: float = 1.2
    locality: float = 0.5  # "grouped": chance a group lands on the token's own rank
    group: int = 4         # "grouped": experts per group
    extra_f32_cols: Tuple[int, ...] = ()   # extra fp32 payloads, columns each
    seed: int = 0

    @property
    def e_local(self) -> int:
        return self.E // self.W

    @property
    def pad_rows(self) -> int:
        """Padding rows per rank: exactly round(pad_frac * T), halves rounded up."""
        return int(np.floor(self.pad_frac * self.T + 0.5))


# The five workloads.
SPECS = {
    1: WorkloadSpec("tiny-w2-e8-k2-t16-h128", W=2, E=8, K=2, T=16, h=128,
                    ids="uniform", pad_frac=0.125, seed=1001),
    2: WorkloadSpec("decode-w8-e64-k8-t128-h2048", W=8, E=64, K=8, T=128, h=2048,
                    ids="uniform", pad_frac=0.05, seed=1002),
    3: WorkloadSpec("prefill-w8-e256-k8-t1024-h7168", W=8, E=256, K=8, T=1024, h=7168,
                    ids="uniform", pad_frac=0.0, seed=1003),
    4: WorkloadSpec("zipf-w16-e128-k8-t512-h4096-scales32", W=16, E=128, K=8, T=512, h=4096,
                    ids="zipf", zipf_s=1.2, extra_f32_cols=(32,), seed=1004),
    5: WorkloadSpec("grouped-w32-e256-k8-t256-h7168", W=32, E=256, K=8, T=256, h=7168,
                    ids="grouped", locality=0.5, group=4,
                    pad_frac=0.15, seed=1005),
}


def spec(cfg: int, **overrides) -> WorkloadSpec:
    """The named workload ``cfg`` (1..5), optionally with fields replaced (e.g. a smaller T)."""
    s = SPECS[cfg]
    if overrides:
        d = dict(s.__dict__)
        d.update(overrides)
        s = WorkloadSpec(**d)
    return s


@dataclass
class Workload:
    spec: WorkloadSpec
    a1: np.ndarray            # [W,T,h] uint16 (bf16 bits)
    topk_ids: np.ndarray      # [W,T,K] int32
    topk_weights: np.ndarray  # [W,T,K] float32
    num_tokens: np.ndarray    # [W] int32
    extras: List[np.ndarray] = field(default_factory=list)  # each [W,T,bytes] uint8

    @property
    def extra_row_bytes(self) -> List[int]:
        return [int(x.shape[2]) for x in self.extras]


def _uniform_ids(rng, n, E, K):
    keys = rng.random((n, E))
    return np.argsort(keys, axis=1, kind="stable")[:, :K]


def _zipf_ids(rng, n, E, K, s):
    # Sampling K distinct experts without replacement, P(e) ~ (e+1)^-s, by
    # Gumbel-top-k: order of the keys log p_e + Gumbel noise, largest first.
    logp = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
    keys = logp[None, :] + rng.gumbel(size=(n, E))
    return np.argsort(-keys, axis=1, kind="stable")[:, :K]


def _grouped_ids(rng, W, T, E, K, group, locality):
    # K/group groups per token; each group picks a rank: the token's own rank
    # with probability `locality`, else a uniform other rank. A group takes
    # `group` distinct experts of its rank. Groups that pick the same rank
    # take consecutive chunks of one random permutation of that rank's
    # experts, so the ids of a token are always distinct.
    e_local = E // W
    n_groups = K // group
    assert n_groups * group == K and e_local >= K
    n = W * T
    home = np.repeat(np.arange(W), T)                      # [n]
    ranks = np.empty((n, n_groups), dtype=np.int64)
    for g in range(n_groups):
        stay = rng.random(n) < locality
        other = rng.integers(0, W - 1, size=n)
        other = other + (other >= home)                    # uniform over ranks != home
        ranks[:, g] = np.where(stay, home, other)
    perm = np.argsort(rng.random((n, n_groups, e_local)), axis=2, kind="stable")
    rows = np.arange(n)
    ids = np.empty((n, K), dtype=np.int64)
    for g in range(n_groups):
        same = ranks[:, :g + 1] == ranks[:, g:g + 1]       # [n, g+1]
        first = np.argmax(same, axis=1)                    # first group on this rank
        used = same[:, :g].sum(axis=1)                     # earlier groups on this rank
        for c in range(group):
            ids[:, g * group + c] = ranks[:, g] * e_local + perm[rows, first, used * group + c]
    return ids


def make(cfg_or_spec, *, num_tokens: Optional[np.ndarray] = None, seed: Optional[int] = None) -> Workload:
    """Draw the workload for a config number or a :class:`WorkloadSpec`.

    ``num_tokens`` optionally gives a ragged batch (tokens per rank, each <= T);
    rows at or beyond a rank's count still hold drawn values but take no part.
    """
    s = spec(cfg_or_spec) if isinstance(cfg_or_spec, int) else cfg_or_spec
    rng = np.random.Generator(np.random.PCG64(s.seed if seed is None else seed))
    W, T, K, E, h = s.W, s.T, s.K, s.E, s.h
    a1 = f32_to_bf16_bits(rng.standard_normal((W, T, h), dtype=np.float32))
    n = W * T
    if s.ids == "uniform":
        ids = _uniform_ids(rng, n, E, K)
    elif s.ids == "zipf":
        ids = _zipf_ids(rng, n, E, K, s.zipf_s)
    elif s.ids == "grouped":
        ids = _grouped_ids(rng, W, T, E, K, s.group, s.locality)
    else:
        raise ValueError(s.ids)
    ids = ids.reshape(W, T, K).astype(np.int32)
    if s.pad_rows:
        for r in range(W):
            rows = rng.choice(T, size=s.pad_rows, replace=False)
            ids[r, rows, :] = -1
    logits = rng.standard_normal((W, T, K), dtype=np.float32)
    ex = np.exp(logits - logits.max(axis=2, keepdims=True), dtype=np.float32)
    w = (ex / ex.sum(axis=2, keepdims=True, dtype=np.float32)).astype(np.float32)
    extras = []
    for cols in s.extra_f32_cols:
        x = rng.uniform(0.5, 2.0, size=(W, T, cols)).astype(np.float32)
        extras.append(np.ascontiguousarray(x).view(np.uint8).reshape(W, T, cols * 4))
    if num_tokens is None:
        nt = np.full(W, T, dtype=np.int32)
    else:
        nt = np.asarray(num_tokens, dtype=np.int32).reshape(W)
    return Workload(s, np.ascontiguousarray(a1), np.ascontiguousarray(ids),
                    np.ascontiguousarray(w), nt, extras)
