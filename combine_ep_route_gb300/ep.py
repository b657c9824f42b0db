"""Torch-facing binding of the EP dispatch/combine library.

``EpContext.dispatch`` and ``EpContext.combine`` pass tensor pointers and the
current CUDA stream to ``ep_dispatch`` / ``ep_combine`` (include/ep.h); PyTorch
provides device memory and streams only. Semantics follow vLLM
``AllToAllBatchedPrepareAndFinalize`` (``capacities``, ``prepare``,
``finalize``) for W expert-parallel ranks held as blocks of one GPU's memory,
with FlashInfer ``MoeAlltoAll``'s extra dispatch payloads and its
dispatch-then-combine state rule.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import torch

from . import _lib as L


@dataclass(frozen=True)
class EpConfig:
    W: int
    E: int
    top_k: int
    max_tokens: int
    hidden: int
    extra_row_bytes: Tuple[int, ...] = ()
    zero_pad: bool = False
    sendbuf: bool = False
    weight_on_input: bool = False   # apply_router_weight_on_input (top_k == 1)
    x_dtype: str = "bf16"           # dispatched rows: "bf16", "fp8" or "fp4x2" (packed pairs)

    @property
    def x_row_bytes(self) -> int:
        return {"bf16": 2 * self.hidden, "fp8": self.hidden, "fp4x2": self.hidden // 2}[self.x_dtype]

    @property
    def x_torch_dtype(self):
        """Torch dtype of a1 / b_a1 rows (packed fp4 rows are uint8 bytes)."""
        return {"bf16": torch.bfloat16, "fp8": torch.float8_e4m3fn, "fp4x2": torch.uint8}[self.x_dtype]

    @property
    def x_row_elems(self) -> int:
        return self.hidden if self.x_dtype != "fp4x2" else self.hidden // 2

    @property
    def e_local(self) -> int:
        return self.E // self.W

    def to_c(self) -> L.EpConfigC:
        c = L.EpConfigC()
        c.W, c.E, c.top_k, c.max_tokens, c.hidden = self.W, self.E, self.top_k, self.max_tokens, self.hidden
        c.x_dtype = {"bf16": L.EP_BF16, "fp8": L.EP_FP8, "fp4x2": L.EP_FP4X2}[self.x_dtype]
        c.n_extra = len(self.extra_row_bytes)
        for i, b in enumerate(self.extra_row_bytes):
            c.extra_row_bytes[i] = int(b)
        c.flags = ((L.EP_FLAG_ZERO_PAD if self.zero_pad else 0) | (L.EP_FLAG_SENDBUF if self.sendbuf else 0)
                   | (L.EP_FLAG_WEIGHT_ON_INPUT if self.weight_on_input else 0))
        return c


def capacities(cfg: EpConfig) -> Tuple[int, int, int]:
    """(token slots per rank, expert slots per token, rows per expert)."""
    a, b, c = C.c_int32(), C.c_int32(), C.c_int32()
    L.check(L.lib().ep_capacities(C.byref(cfg.to_c()), C.byref(a), C.byref(b), C.byref(c)),
            "ep_capacities")
    return a.value, b.value, c.value


def workspace_bytes(cfg: EpConfig) -> int:
    n = C.c_size_t()
    L.check(L.lib().ep_workspace_bytes(C.byref(cfg.to_c()), C.byref(n)), "ep_workspace_bytes")
    return n.value


def _stream_ptr(stream: Optional[torch.cuda.Stream], dev: torch.device) -> int:
    """The stream to enqueue on. The library launches on the current device, so
    that must be the device the buffers live on, and a given stream must belong
    to it: otherwise the kernels would address another device's memory."""
    cur = torch.cuda.current_device()
    if dev.index != cur:
        raise ValueError(f"the buffers are on {dev} but the current device is cuda:{cur}; "
                         f"make {dev} current (torch.cuda.set_device) first")
    s = stream if stream is not None else torch.cuda.current_stream()
    if s.device.index != cur:
        raise ValueError(f"stream is on {s.device}, the buffers on {dev}")
    return s.cuda_stream


def _cuda_device(device) -> torch.device:
    """A CUDA device with its index filled in (the current device when absent)."""
    d = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if d.type != "cuda":
        raise ValueError(f"want a CUDA device, got {d}")
    return d if d.index is not None else torch.device("cuda", torch.cuda.current_device())


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape: Sequence[int], dev) -> None:
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or t.device != dev:
        raise ValueError(f"{name}: want contiguous {dtype} {tuple(shape)} on {dev}, got "
                         f"{t.dtype} {tuple(t.shape)} on {t.device} (contiguous={t.is_contiguous()})")


@dataclass
class DispatchOut:
    b_a1: torch.Tensor                 # [W, e_local, Ecap, h] bf16
    expert_num_tokens: torch.Tensor    # [W, e_local] int32
    extra_out: List[torch.Tensor] = field(default_factory=list)  # [W, e_local, Ecap, bytes] uint8


class EpContext:
    """A dispatch/combine context over a workspace allocated through PyTorch, or
    over ``workspace`` (a contiguous uint8 device tensor of at least
    ``workspace_bytes(cfg)`` bytes, 256-byte aligned) that the caller owns."""

    def __init__(self, cfg: EpConfig, device: Optional[torch.device] = None,
                 workspace: Optional[torch.Tensor] = None):
        self.cfg = cfg
        self.device = _cuda_device(device)
        self.tok_cap, self.slots, self.expert_cap = capacities(cfg)
        nbytes = workspace_bytes(cfg)
        if workspace is None:
            self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        else:
            if (workspace.dtype != torch.uint8 or not workspace.is_contiguous() or workspace.numel() < nbytes
                    or workspace.device != self.device):
                raise ValueError(f"workspace: want a contiguous uint8 tensor of at least {nbytes} bytes "
                                 f"on {self.device}")
            self.workspace = workspace[:nbytes]
        h = C.c_void_p()
        L.check(L.lib().ep_ctx_create(C.byref(cfg.to_c()), C.c_void_p(self.workspace.data_ptr()),
                                      nbytes, C.byref(h)), "ep_ctx_create")
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            try:
                L.lib().ep_ctx_destroy(h)
            except Exception:
                pass
            self._h = None

    # ------------------------------------------------------------ buffers
    def alloc_dispatch_outputs(self) -> DispatchOut:
        c = self.cfg
        b = torch.empty((c.W, c.e_local, self.expert_cap, c.x_row_elems), dtype=c.x_torch_dtype,
                        device=self.device)
        n = torch.empty((c.W, c.e_local), dtype=torch.int32, device=self.device)
        ex = [torch.empty((c.W, c.e_local, self.expert_cap, nb), dtype=torch.uint8, device=self.device)
              for nb in c.extra_row_bytes]
        return DispatchOut(b, n, ex)

    # ----------------------------------------------------------- the path
    def dispatch(self, a1: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                 num_tokens: Optional[torch.Tensor] = None, extras: Sequence[torch.Tensor] = (),
                 out: Optional[DispatchOut] = None, path: str = "fused",
                 stream: Optional[torch.cuda.Stream] = None) -> DispatchOut:
        """Route, deduplicate, slot and deliver all W ranks' tokens (``prepare``)."""
        c, dev = self.cfg, self.device
        _need(a1, "a1", c.x_torch_dtype, (c.W, c.max_tokens, c.x_row_elems), dev)
        _need(topk_ids, "topk_ids", torch.int32, (c.W, c.max_tokens, c.top_k), dev)
        _need(topk_weights, "topk_weights", torch.float32, (c.W, c.max_tokens, c.top_k), dev)
        if num_tokens is not None:
            _need(num_tokens, "num_tokens", torch.int32, (c.W,), dev)
        if len(extras) != len(c.extra_row_bytes):
            raise ValueError(f"want {len(c.extra_row_bytes)} extra payloads, got {len(extras)}")
        for i, (x, nb) in enumerate(zip(extras, c.extra_row_bytes)):
            if not x.is_contiguous() or x.device != dev or x.numel() * x.element_size() != c.W * c.max_tokens * nb:
                raise ValueError(f"extras[{i}]: want contiguous [W, Tm, {nb} bytes] on {dev}")
        if out is None:
            out = self.alloc_dispatch_outputs()
        _need(out.b_a1, "b_a1", c.x_torch_dtype, (c.W, c.e_local, self.expert_cap, c.x_row_elems), dev)
        _need(out.expert_num_tokens, "expert_num_tokens", torch.int32, (c.W, c.e_local), dev)
        n_ex = len(c.extra_row_bytes)
        ein = (C.c_void_p * max(n_ex, 1))(*[x.data_ptr() for x in extras])
        eout = (C.c_void_p * max(n_ex, 1))(*[x.data_ptr() for x in out.extra_out])
        p = {"fused": L.EP_PATH_FUSED, "sendbuf": L.EP_PATH_SENDBUF}[path]
        rc = L.lib().ep_dispatch(self._h, a1.data_ptr(),
                                 None if num_tokens is None else num_tokens.data_ptr(),
                                 topk_ids.data_ptr(), topk_weights.data_ptr(),
                                 ein if n_ex else None, out.b_a1.data_ptr(),
                                 eout if n_ex else None, out.expert_num_tokens.data_ptr(), p,
                                 _stream_ptr(stream, dev))
        L.check(rc, "ep_dispatch")
        return out

    def combine(self, expert_out: torch.Tensor, out: Optional[torch.Tensor] = None,
                out_dtype: torch.dtype = torch.bfloat16,
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """Weighted fp32 sum of each token's expert rows (``finalize``)."""
        c, dev = self.cfg, self.device
        _need(expert_out, "expert_out", torch.bfloat16, (c.W, c.e_local, self.expert_cap, c.hidden), dev)
        if out is None:
            out = torch.empty((c.W, c.max_tokens, c.hidden), dtype=out_dtype, device=dev)
        _need(out, "out", out_dtype, (c.W, c.max_tokens, c.hidden), dev)
        code = {torch.bfloat16: L.EP_BF16, torch.float32: L.EP_F32}[out_dtype]
        L.check(L.lib().ep_combine(self._h, expert_out.data_ptr(), code, out.data_ptr(),
                                   _stream_ptr(stream, dev)), "ep_combine")
        return out

    def combine_two_stage(self, expert_out: torch.Tensor, out: Optional[torch.Tensor] = None,
                          out_dtype: torch.dtype = torch.bfloat16,
                          stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
        """``finalize`` in the page's two-stage rounding (needs ``sendbuf=True``)."""
        c, dev = self.cfg, self.device
        _need(expert_out, "expert_out", torch.bfloat16, (c.W, c.e_local, self.expert_cap, c.hidden), dev)
        if out is None:
            out = torch.empty((c.W, c.max_tokens, c.hidden), dtype=out_dtype, device=dev)
        _need(out, "out", out_dtype, (c.W, c.max_tokens, c.hidden), dev)
        code = {torch.bfloat16: L.EP_BF16, torch.float32: L.EP_F32}[out_dtype]
        L.check(L.lib().ep_combine_two_stage(self._h, expert_out.data_ptr(), code, out.data_ptr(),
                                             _stream_ptr(stream, dev)), "ep_combine_two_stage")
        return out

    # ---------------------------------------------------------- utilities
    def status(self, stream: Optional[torch.cuda.Stream] = None) -> int:
        """Synchronise and return the device status code (0 = ok); clears it."""
        return int(L.lib().ep_status(self._h, _stream_ptr(stream, self.device)))

    def check(self, stream: Optional[torch.cuda.Stream] = None) -> None:
        L.check(self.status(stream), "device status")

    def reset(self) -> None:
        L.check(L.lib().ep_ctx_reset(self._h), "ep_ctx_reset")

    def set_option(self, option: int, value: int) -> None:
        L.check(L.lib().ep_set_option(self._h, option, int(value)), "ep_set_option")

    def kernel_times(self) -> Dict[str, Tuple[int, float, int]]:
        """{kernel: (launches, summed event ms, timed launches)} since the last read."""
        kt = L.EpKernelTimesC()
        L.check(L.lib().ep_kernel_times(self._h, C.byref(kt)), "ep_kernel_times")
        return {n: (kt.launches[i], kt.total_ms[i], kt.timed[i]) for i, n in enumerate(L.KERNEL_NAMES)}

    def metadata(self) -> Dict[str, torch.Tensor]:
        """Views of the routing metadata in the workspace (see ep_metadata_t)."""
        m = L.EpMetadataC()
        L.check(L.lib().ep_get_metadata(self._h, C.byref(m)), "ep_get_metadata")
        c = self.cfg
        W, T, K, S = c.W, c.max_tokens, c.top_k, m.slots_per_token
        base = self.workspace.data_ptr()

        def view(ptr, n, dtype, shape):
            off = ptr - base
            esz = torch.tensor([], dtype=dtype).element_size()
            return self.workspace[off:off + n * esz].view(dtype).view(*shape)

        out = {
            "send_cnt": view(m.send_cnt, W * W, torch.int32, (W, W)),
            "pair_row": view(m.pair_row, W * T * K, torch.int32, (W, T, K)),
            "pair_w": view(m.pair_w, W * T * K, torch.float32, (W, T, K)),
            "pair_send": view(m.pair_send, W * T * K, torch.int32, (W, T, K)),
            "recv_eloc": view(m.recv_eloc, W * W * T * S, torch.int32, (W, W, T, S)),
            "recv_w": view(m.recv_w, W * W * T * S, torch.float32, (W, W, T, S)),
            "recv_row": view(m.recv_row, W * W * T * S, torch.int32, (W, W, T, S)),
        }
        if m.send_x:
            rb = m.row_bytes
            out["send_x"] = view(m.send_x, W * W * T * rb, torch.uint8, (W, W, T, rb))
            out["recv_x"] = view(m.recv_x, W * W * T * rb, torch.uint8, (W, W, T, rb))
        return out


# ------------------------------------------------- all-gather / reduce-scatter

@dataclass
class AgrsBuffers:
    """Device buffers of ``ep_agrs`` (see ep_agrs_buffers_t)."""
    x_g: torch.Tensor      # [W, W*Tm, h] bf16: every rank's gathered token rows
    ids_g: torch.Tensor    # [W, W*Tm, K] int32
    w_g: torch.Tensor      # [W, W*Tm, K] float32
    y: torch.Tensor        # [W, W*Tm, h] bf16: each rank's expert output per gathered token
    status: torch.Tensor   # [1] int32: first device-side EP_ERR_* of the last call, 0 if none

    def to_c(self) -> L.EpAgrsBuffersC:
        b = L.EpAgrsBuffersC()
        b.x_g, b.ids_g, b.w_g = self.x_g.data_ptr(), self.ids_g.data_ptr(), self.w_g.data_ptr()
        b.y, b.status = self.y.data_ptr(), self.status.data_ptr()
        return b


def alloc_agrs_buffers(cfg: EpConfig, device) -> AgrsBuffers:
    W, T, K, h = cfg.W, cfg.max_tokens, cfg.top_k, cfg.hidden
    dev = torch.device(device)
    return AgrsBuffers(
        x_g=torch.empty(W, W * T, h, dtype=torch.bfloat16, device=dev),
        ids_g=torch.empty(W, W * T, K, dtype=torch.int32, device=dev),
        w_g=torch.empty(W, W * T, K, dtype=torch.float32, device=dev),
        y=torch.empty(W, W * T, h, dtype=torch.bfloat16, device=dev),
        status=torch.zeros(1, dtype=torch.int32, device=dev))


def agrs(cfg: EpConfig, a1: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
         num_tokens: Optional[torch.Tensor] = None, out_dtype: torch.dtype = torch.bfloat16,
         buffers: Optional[AgrsBuffers] = None, out: Optional[torch.Tensor] = None,
         stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """The all-gather / reduce-scatter route with identity experts (``ep_agrs``):
    returns out [W, Tm, h] in ``out_dtype``. Device-side errors land in
    ``buffers.status`` (read it after synchronising)."""
    W, T, K, h = cfg.W, cfg.max_tokens, cfg.top_k, cfg.hidden
    dev = a1.device
    _need(a1, "a1", torch.bfloat16, (W, T, h), dev)
    _need(topk_ids, "topk_ids", torch.int32, (W, T, K), dev)
    _need(topk_weights, "topk_weights", torch.float32, (W, T, K), dev)
    if num_tokens is not None:
        _need(num_tokens, "num_tokens", torch.int32, (W,), dev)
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("out_dtype must be bfloat16 or float32")
    if buffers is None:
        buffers = alloc_agrs_buffers(cfg, dev)
    if out is None:
        out = torch.empty(W, T, h, dtype=out_dtype, device=dev)
    _need(out, "out", out_dtype, (W, T, h), dev)
    L.check(L.lib().ep_agrs(C.byref(cfg.to_c()),
                            num_tokens.data_ptr() if num_tokens is not None else None,
                            a1.data_ptr(), topk_ids.data_ptr(), topk_weights.data_ptr(),
                            C.byref(buffers.to_c()),
                            L.EP_F32 if out_dtype == torch.float32 else L.EP_BF16,
                            out.data_ptr(), _stream_ptr(stream, dev)), "ep_agrs")
    return out
