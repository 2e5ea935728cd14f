"""DeepEP-style ``Buffer`` over the C ABI: the call shapes of
low_latency_dispatch(hidden_states, topk_idx, num_max_dispatch_tokens_per_rank,
num_experts) and low_latency_combine(hidden_states, topk_idx, topk_weights,
handle, num_experts) from "如何突破MoE通信瓶颈：DeepEP跨节点优化技术终极指南"
(section 核心API示例), the preallocated buffer of ``low_latency_mode=True``
and the size hint ``get_low_latency_rdma_size_hint()`` (section
低延迟模式关键特性 / 内存优化).

All R expert-parallel ranks are virtual ranks on this GPU: ``hidden_states``
is every rank's tokens, [R, T, H] bf16, and ``topk_idx`` is [R, T, K] int64.
"""
from __future__ import annotations

import torch

from . import ep


class Handle:
    """A cached dispatch layout (owned device buffers of libep)."""

    def __init__(self, buf: "Buffer"):
        self._buf = buf
        self._h = ep.ep_handle_create(buf._ctx)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            try:
                ep.ep_handle_destroy(h)
            except Exception:
                pass
            self._h = None

    @property
    def raw(self):
        return self._h

    def info(self) -> ep.ep_handle_info:
        return ep.ep_handle_get_info(self._h)

    def tensors(self) -> dict:
        """The layout arrays (slot, src_info, cnt_er, off_er, base,
        tokens_per_expert) as CUDA tensors viewing the handle's memory."""
        info = self.info()
        b = self._buf
        N = max(info.num_tokens, 0)
        return dict(
            slot=_device_view(info.slot, (N, b.topk), "<i4"),
            src_info=_device_view(info.src_info, (info.rows,), "<i4"),
            cnt_er=_device_view(info.cnt_er, (b.num_experts, b.num_ranks), "<i4"),
            off_er=_device_view(info.off_er, (b.num_experts, b.num_ranks), "<i4"),
            base=_device_view(info.base, (b.num_experts,), "<i8"),
            tokens_per_expert=_device_view(info.tokens_per_expert, (b.num_experts,), "<i4"),
        )


class _DeviceArray:
    """Minimal __cuda_array_interface__ exporter for a raw device pointer."""

    def __init__(self, ptr: int, shape: tuple, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (int(ptr or 0), False), "version": 3,
                                         "strides": None}


def _device_view(ptr: int, shape: tuple, typestr: str) -> torch.Tensor:
    dtype = {"<i4": torch.int32, "<i8": torch.int64}[typestr]
    if not ptr or 0 in shape:
        return torch.empty(shape, dtype=dtype, device="cuda")
    return torch.as_tensor(_DeviceArray(ptr, shape, typestr), device="cuda")


class Buffer:
    """One expert-parallel group of ``num_ranks`` virtual ranks.

    ``low_latency_mode=True`` gives the padded layout (E fixed buffers of
    R*num_max_dispatch_tokens_per_rank rows); False gives the packed layout
    of the normal (high-throughput) kernels.  ``max_sms`` caps the SMs the
    dispatch / combine kernels use (0 = all)."""

    def __init__(self, num_ranks: int, num_max_dispatch_tokens_per_rank: int, hidden: int,
                 num_experts: int, num_topk: int, low_latency_mode: bool = True, max_sms: int = 0,
                 num_hook_sms: int = 0):
        self.num_ranks = num_ranks
        self.max_tokens_per_rank = num_max_dispatch_tokens_per_rank
        self.hidden = hidden
        self.num_experts = num_experts
        self.topk = num_topk
        self.low_latency_mode = low_latency_mode
        self.cfg = ep.make_config(num_ranks, num_max_dispatch_tokens_per_rank, hidden, num_experts,
                                  num_topk, ep.EP_LAYOUT_PADDED if low_latency_mode else ep.EP_LAYOUT_PACKED,
                                  max_sms)
        self._ctx = ep.ep_create(self.cfg)
        self.rows = ep.ep_recv_rows(self.cfg)
        self.num_hook_sms = num_hook_sms   # SMs of the receive hooks' copy kernels (0: max_sms / all)
        self._send = {}                    # send / staging buffers of the split calls, made on first use

    def __del__(self):
        ctx = getattr(self, "_ctx", None)
        if ctx is not None and ctx.value:
            try:
                ep.ep_destroy(ctx)
            except Exception:
                pass
            self._ctx = None

    @property
    def ctx(self):
        return self._ctx

    # -------------------------------------------------------- sizes
    @staticmethod
    def get_low_latency_rdma_size_hint(num_max_dispatch_tokens_per_rank: int, hidden: int,
                                       num_ranks: int, num_experts: int, num_topk: int = 8,
                                       use_fp8: bool = True) -> int:
        """Bytes of receive buffers (payload + FP8 scales) for the padded layout."""
        cfg = ep.make_config(num_ranks, num_max_dispatch_tokens_per_rank, hidden, num_experts, num_topk)
        payload, scales = ep.ep_recv_bytes(cfg, use_fp8)
        return payload + scales

    def alloc_recv(self, use_fp8: bool):
        """Allocate receive buffers: (recv_x, recv_scales or None)."""
        dev = torch.device("cuda", torch.cuda.current_device())
        if use_fp8:
            return (torch.empty(self.rows, self.hidden, dtype=torch.float8_e4m3fn, device=dev),
                    torch.empty(self.rows, self.hidden // 128, dtype=torch.float32, device=dev))
        return torch.empty(self.rows, self.hidden, dtype=torch.bfloat16, device=dev), None

    def new_handle(self) -> Handle:
        return Handle(self)

    @property
    def rank_rows(self) -> int:
        """Rows of a rank-deduplicated receive buffer (ep_rank_recv_rows)."""
        return ep.ep_rank_recv_rows(self.cfg)

    def alloc_rank_recv(self, use_fp8: bool):
        """Receive buffers for the rank-deduplicated layout: (recv_x, recv_scales or None)."""
        dev = torch.device("cuda", torch.cuda.current_device())
        rows = self.rank_rows
        if use_fp8:
            return (torch.empty(rows, self.hidden, dtype=torch.float8_e4m3fn, device=dev),
                    torch.empty(rows, self.hidden // 128, dtype=torch.float32, device=dev))
        return torch.empty(rows, self.hidden, dtype=torch.bfloat16, device=dev), None

    def get_rank_layout(self, topk_idx: torch.Tensor, topk_weights: torch.Tensor | None = None,
                        handle: Handle | None = None):
        """Rank-deduplicated (normal-mode) layout: (num_tokens_per_rank [R],
        recv_topk_idx [rows, K] local expert ids or -1, recv_topk_weights
        [rows, K], handle).  The handle then serves low_latency_dispatch
        (topk_idx=None, buffers from alloc_rank_recv) and low_latency_combine
        (topk_weights=None: the expert side applies the weights)."""
        T = self._tokens_per_rank(topk_idx)
        dev = topk_idx.device
        ntr = torch.empty(self.num_ranks, dtype=torch.int32, device=dev)
        rows = self.rank_rows
        ridx = torch.empty(rows, self.topk, dtype=torch.int32, device=dev)
        rw = torch.empty(rows, self.topk, dtype=torch.float32, device=dev)
        handle = handle or Handle(self)
        w = None if topk_weights is None else topk_weights.reshape(-1, self.topk)
        ep.ep_get_rank_layout(self._ctx, topk_idx, w, T, ntr, ridx, rw, handle.raw)
        return ntr, ridx, rw, handle

    # -------------------------------------------------------- operations
    def _tokens_per_rank(self, topk_idx: torch.Tensor) -> int:
        if topk_idx.dim() != 3 or topk_idx.shape[0] != self.num_ranks or topk_idx.shape[2] != self.topk:
            raise ValueError(f"topk_idx must be [R={self.num_ranks}, T, K={self.topk}]")
        return topk_idx.shape[1]

    def get_dispatch_layout(self, topk_idx: torch.Tensor, handle: Handle | None = None):
        """(num_tokens_per_rank [R], num_tokens_per_expert [E],
        is_token_in_rank [R*T, R] bool, handle)."""
        T = self._tokens_per_rank(topk_idx)
        dev = topk_idx.device
        ntr = torch.empty(self.num_ranks, dtype=torch.int32, device=dev)
        nte = torch.empty(self.num_experts, dtype=torch.int32, device=dev)
        itr = torch.empty(self.num_ranks * T, self.num_ranks, dtype=torch.bool, device=dev)
        handle = handle or Handle(self)
        ep.ep_get_dispatch_layout(self._ctx, topk_idx, T, ntr, nte, itr, handle.raw)
        return ntr, nte, itr, handle

    def _send_buffers(self, key: str, use_fp8: bool):
        """Send buffer of a split dispatch ([R*Tmax, H] + scales) or staging
        buffer of a split combine ([R*Tmax*K, H] bf16), kept for reuse."""
        k = (key, use_fp8)
        if k not in self._send:
            dev = torch.device("cuda", torch.cuda.current_device())
            n = self.num_ranks * self.max_tokens_per_rank
            if key == "dispatch":
                x = torch.empty(n, self.hidden, dtype=torch.float8_e4m3fn if use_fp8 else torch.bfloat16, device=dev)
                sc = torch.empty(n, self.hidden // 128, dtype=torch.float32, device=dev) if use_fp8 else None
                self._send[k] = (x, sc)
            else:
                self._send[k] = (torch.empty(n * self.topk, self.hidden, dtype=torch.bfloat16, device=dev), None)
        return self._send[k]

    def low_latency_dispatch(self, hidden_states: torch.Tensor, topk_idx: torch.Tensor | None,
                             num_max_dispatch_tokens_per_rank: int, num_experts: int,
                             use_fp8: bool = True, handle: Handle | None = None,
                             out=None, recv_count: torch.Tensor | None = None,
                             return_recv_hook: bool = False):
        """Returns ((recv_x, recv_scales) if use_fp8 else recv_x, recv_count, handle).
        topk_idx=None reuses the layout cached in ``handle``.  With
        return_recv_hook=True only the send half runs now and a fourth value,
        ``hook``, is returned: calling it enqueues the receive (copy-engine
        copies on ``num_hook_sms`` SMs); the receive buffers and counts hold
        their values once the hook's work has run."""
        if num_max_dispatch_tokens_per_rank != self.max_tokens_per_rank or num_experts != self.num_experts:
            raise ValueError("num_max_dispatch_tokens_per_rank / num_experts differ from the Buffer's")
        T = hidden_states.numel() // (self.num_ranks * self.hidden)
        if hidden_states.numel() != self.num_ranks * T * self.hidden:
            raise ValueError("hidden_states must be [R, T, H]")
        if topk_idx is not None and self._tokens_per_rank(topk_idx) != T:
            raise ValueError("topk_idx and hidden_states disagree on T")
        if topk_idx is None and handle is None:
            raise ValueError("reusing a layout needs a handle")
        handle = handle or Handle(self)
        recv_x, recv_scales = out if out is not None else self.alloc_recv(use_fp8)
        if recv_count is None:
            recv_count = torch.empty(self.num_experts, dtype=torch.int32, device=hidden_states.device)
        if return_recv_hook:
            send_x, send_sc = (hidden_states, None) if not use_fp8 else self._send_buffers("dispatch", True)
            ep.ep_dispatch_send(self._ctx, hidden_states, topk_idx, T, use_fp8, handle.raw, send_x, send_sc)
            sc = recv_scales if use_fp8 else None
            hook_sms = self.num_hook_sms

            def hook(stream=None):
                ep.ep_dispatch_recv(self._ctx, handle.raw, use_fp8, send_x, send_sc, recv_x, sc, recv_count,
                                    hook_sms, stream)
            return ((recv_x, recv_scales) if use_fp8 else recv_x), recv_count, handle, hook
        ep.ep_dispatch(self._ctx, hidden_states, topk_idx, T, use_fp8, handle.raw,
                       recv_x, recv_scales if use_fp8 else None, recv_count)
        return ((recv_x, recv_scales) if use_fp8 else recv_x), recv_count, handle

    def low_latency_combine(self, hidden_states: torch.Tensor, topk_idx: torch.Tensor | None,
                            topk_weights: torch.Tensor | None, handle: Handle, num_experts: int,
                            out: torch.Tensor | None = None, return_recv_hook: bool = False):
        """Weighted top-k reduce of expert outputs ``hidden_states`` [rows, H]
        bf16 (receive layout of ``handle``) back to [R*T, H] bf16 tokens.
        ``topk_idx`` is accepted for call compatibility; the handle's slots
        decide which rows are read.  topk_weights=None means all ones.  With
        return_recv_hook=True the expert outputs are sent back now (copy
        engine) and (out, hook) is returned: calling hook enqueues the
        reduce."""
        if num_experts != self.num_experts:
            raise ValueError("num_experts differs from the Buffer's")
        info = handle.info()
        if info.tokens_per_rank < 0:
            raise ep.EPError(ep.EP_ERR_NO_LAYOUT, "low_latency_combine")
        N = info.num_tokens
        if out is None:
            out = torch.empty(N, self.hidden, dtype=torch.bfloat16, device=hidden_states.device)
        if return_recv_hook:
            send_y, _ = self._send_buffers("combine", False)
            ep.ep_combine_send(self._ctx, handle.raw, hidden_states, send_y, self.num_hook_sms)

            def hook(stream=None):
                ep.ep_combine_recv(self._ctx, handle.raw, send_y, topk_weights, out, stream)
            return out, hook
        ep.ep_combine(self._ctx, hidden_states, topk_weights, handle.raw, out)
        return out

    def _rank_buffers(self, key: str, use_fp8: bool, wire: int):
        """Send buffer of the rank transport ([ep_rank_send_rows, H] + scales,
        or bf16 for the combine) and, for the host wire, its pinned staging
        buffer; kept for reuse."""
        k = ("rank", key, use_fp8)
        if k not in self._send:
            dev = torch.device("cuda", torch.cuda.current_device())
            n = ep.ep_rank_send_rows(self.cfg)
            fp8 = use_fp8 and key == "dispatch"
            x = torch.empty(n, self.hidden, dtype=torch.float8_e4m3fn if fp8 else torch.bfloat16, device=dev)
            sc = torch.empty(n, self.hidden // 128, dtype=torch.float32, device=dev) if fp8 else None
            self._send[k] = (x, sc)
        x, sc = self._send[k]
        stage = None
        if wire == ep.EP_WIRE_HOST:
            ks = ("rank_stage",)
            if ks not in self._send:
                n = ep.ep_rank_send_rows(self.cfg)
                self._send[ks] = torch.empty(n * (2 * self.hidden + self.hidden // 32), dtype=torch.uint8).pin_memory()
            stage = self._send[ks]
        return x, sc, stage

    def rank_dispatch(self, hidden_states: torch.Tensor, topk_idx: torch.Tensor | None,
                      topk_weights: torch.Tensor | None = None, use_fp8: bool = False,
                      handle: Handle | None = None, wire: int = ep.EP_WIRE_DEVICE,
                      return_recv_hook: bool = False):
        """Rank-deduplicated dispatch whose receive runs no kernel: the send
        half (layout, send rows, one cast per token) now, the receive as one
        copy per (source rank, destination rank) run over ``wire``
        (EP_WIRE_DEVICE: device copies at HBM speed; EP_WIRE_HOST: through
        pinned host memory on the copy engines, no SM).  Returns
        ((recv_x, recv_scales) if use_fp8 else recv_x, recv_count [R],
        recv_topk_idx [rows, K], recv_topk_weights [rows, K] (None when the
        layout is reused), handle), plus
        ``hook`` when return_recv_hook is True (the receive is enqueued when
        it is called; otherwise it is enqueued before returning).
        topk_idx=None reuses the layout in ``handle``."""
        T = hidden_states.numel() // (self.num_ranks * self.hidden)
        if hidden_states.numel() != self.num_ranks * T * self.hidden:
            raise ValueError("hidden_states must be [R, T, H]")
        if topk_idx is not None and self._tokens_per_rank(topk_idx) != T:
            raise ValueError("topk_idx and hidden_states disagree on T")
        if topk_idx is None and handle is None:
            raise ValueError("reusing a layout needs a handle")
        handle = handle or Handle(self)
        dev = hidden_states.device
        rows = self.rank_rows
        ridx = torch.empty(rows, self.topk, dtype=torch.int32, device=dev)
        rw = torch.empty(rows, self.topk, dtype=torch.float32, device=dev)
        send_x, send_sc, stage = self._rank_buffers("dispatch", use_fp8, wire)
        w = None if topk_weights is None else topk_weights.reshape(-1, self.topk)
        ep.ep_rank_dispatch_send(self._ctx, hidden_states, topk_idx, w, T, use_fp8,
                                 ridx if topk_idx is not None else None,
                                 rw if topk_idx is not None else None, handle.raw, send_x, send_sc)
        recv_x, recv_scales = self.alloc_rank_recv(use_fp8)
        recv_count = torch.empty(self.num_ranks, dtype=torch.int32, device=dev)

        def hook(stream=None):
            ep.ep_rank_dispatch_recv(self._ctx, handle.raw, use_fp8, send_x, send_sc, recv_x,
                                     recv_scales if use_fp8 else None, recv_count, wire, stage, stream)
        if topk_idx is None:  # a reused layout: the rows' local top-k came with the first call
            ridx = rw = None
        res = (((recv_x, recv_scales) if use_fp8 else recv_x), recv_count, ridx, rw, handle)
        if return_recv_hook:
            return res + (hook,)
        hook()
        return res

    def rank_combine(self, hidden_states: torch.Tensor, handle: Handle, wire: int = ep.EP_WIRE_DEVICE,
                     out: torch.Tensor | None = None, return_recv_hook: bool = False):
        """The rank transport's combine: the expert outputs ``hidden_states``
        (rank receive layout, bf16, local weights already applied) travel back
        over ``wire`` now, and the per-token sum over its rank rows follows
        (in ``hook`` when return_recv_hook is True).  Returns out [R*T, H]
        (and hook)."""
        info = handle.info()
        if info.tokens_per_rank < 0:
            raise ep.EPError(ep.EP_ERR_NO_LAYOUT, "rank_combine")
        if out is None:
            out = torch.empty(info.num_tokens, self.hidden, dtype=torch.bfloat16, device=hidden_states.device)
        send_y, _, stage = self._rank_buffers("combine", False, wire)
        ep.ep_rank_combine_send(self._ctx, handle.raw, hidden_states, send_y, wire, stage)

        def hook(stream=None):
            ep.ep_rank_combine_recv(self._ctx, handle.raw, send_y, out, stream)
        if return_recv_hook:
            return out, hook
        hook()
        return out

    def round_trip(self, hidden_states: torch.Tensor, topk_idx: torch.Tensor | None,
                   topk_weights: torch.Tensor | None, use_fp8: bool = True, chunk_tokens: int = 0,
                   handle: Handle | None = None, recv=None, y: torch.Tensor | None = None,
                   out: torch.Tensor | None = None):
        """Dispatch -> identity expert -> combine over chunks of ``chunk_tokens``
        tokens (0: one chunk, -1: the L2-sized automatic chunk); topk_idx=None
        reuses the layout in ``handle``.  Returns (out [R*T, H] bf16, handle)."""
        T = hidden_states.numel() // (self.num_ranks * self.hidden)
        if hidden_states.numel() != self.num_ranks * T * self.hidden:
            raise ValueError("hidden_states must be [R, T, H]")
        if topk_idx is not None and self._tokens_per_rank(topk_idx) != T:
            raise ValueError("topk_idx and hidden_states disagree on T")
        if topk_idx is None and handle is None:
            raise ValueError("reusing a layout needs a handle")
        handle = handle or Handle(self)
        recv_x, recv_scales = recv if recv is not None else self.alloc_recv(use_fp8)
        dev = hidden_states.device
        if y is None:
            y = recv_x if not use_fp8 else torch.empty(self.rows, self.hidden, dtype=torch.bfloat16, device=dev)
        if out is None:
            out = torch.empty(self.num_ranks * T, self.hidden, dtype=torch.bfloat16, device=dev)
        ep.ep_round_trip(self._ctx, hidden_states, topk_idx, T, topk_weights, use_fp8, handle.raw,
                         recv_x, recv_scales if use_fp8 else None, y, out, chunk_tokens)
        return out, handle

    def device_status(self) -> int:
        """Synchronise the current stream; return and clear the device status."""
        return ep.ep_get_device_status(self._ctx)
