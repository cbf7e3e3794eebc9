"""MoELayer: one MoE expert block on one GPU, driven through the C ABI.

Holds the device weights, the workspace and the output buffers of one layer
and calls moe_fwd / moe_select_retained / moe_bwd. It allocates with torch
(the library itself allocates nothing) and adds no computation of its own.
"""
from __future__ import annotations

import torch

from . import _lib
from .inputs import Workload

WEIGHTS = ["w_router", "w_gate", "w_up", "w_down", "ws_gate", "ws_up", "ws_down"]


class MoELayer:
    def __init__(self, w: Workload, params: dict, device="cuda", record_routing: bool = False,
                 recompute: bool = False):
        """params: CPU or device tensors named as in inputs.make_inputs (weights + optional router_bias).

        recompute: the backward re-derives the expert activations instead of
        using the forward's (the keep-nothing mode, MOE_RECOMPUTE)."""
        self.w = w
        self.device = torch.device(device)
        self.dims = _lib.make_dims(w.T, w.H, w.F, w.E, w.k, w.F_shared, w.dtype, w.frozen, recompute)
        self.io = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        dev = self.device
        self.p = {}
        for n in WEIGHTS + ["router_bias"]:
            t = params.get(n)
            self.p[n] = None if t is None else t.to(dev).contiguous()
        self.ws = _lib.alloc_workspace(self.dims, dev)
        T, H, F, E, k, Fs = w.T, w.H, w.F, w.E, w.k, w.F_shared
        self.y = torch.empty(T, H, dtype=self.io, device=dev)
        self.dx = torch.empty(T, H, dtype=self.io, device=dev)
        self.grads = {}
        if not w.frozen:
            self.grads = dict(
                dw_router=torch.empty(H, E, dtype=self.io, device=dev),
                dw_gate=torch.empty(E, H, F, dtype=self.io, device=dev),
                dw_up=torch.empty(E, H, F, dtype=self.io, device=dev),
                dw_down=torch.empty(E, F, H, dtype=self.io, device=dev),
            )
            if Fs:
                self.grads.update(
                    dws_gate=torch.empty(H, Fs, dtype=self.io, device=dev),
                    dws_up=torch.empty(H, Fs, dtype=self.io, device=dev),
                    dws_down=torch.empty(Fs, H, dtype=self.io, device=dev),
                )
        self.record = record_routing
        if record_routing:
            self.topk_idx = torch.empty(T, k, dtype=torch.int32, device=dev)
            self.topk_w = torch.empty(T, k, dtype=torch.float32, device=dev)
            self.offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
            self.row_of_pair = torch.empty(T * k, dtype=torch.int32, device=dev)
            self.logits = torch.empty(T, E, dtype=torch.float32, device=dev)
            self.ret_offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
            self.ret_rows = torch.full((T * k,), -1, dtype=torch.int32, device=dev)
            self.scores = torch.empty(T * k, dtype=torch.float32, device=dev)

    def forward(self, x: torch.Tensor, stream=None) -> torch.Tensor:
        p = self.p
        r = self.record
        _lib.moe_fwd(self.dims, self.ws, x, p["w_router"], p["router_bias"], p["w_gate"], p["w_up"], p["w_down"],
                     p["ws_gate"], p["ws_up"], p["ws_down"], self.y,
                     self.topk_idx if r else None, self.topk_w if r else None, self.offsets if r else None,
                     self.row_of_pair if r else None, self.logits if r else None, stream=stream)
        return self.y

    def forward_decode(self, x: torch.Tensor, stream=None) -> torch.Tensor:
        """Inference forward through the fused decode kernel (1 <= T <= 16, bf16)."""
        p = self.p
        r = self.record
        _lib.moe_fwd_decode(self.dims, self.ws, x, p["w_router"], p["router_bias"], p["w_gate"], p["w_up"],
                            p["w_down"], p["ws_gate"], p["ws_up"], p["ws_down"], self.y,
                            self.topk_idx if r else None, self.topk_w if r else None, self.logits if r else None,
                            stream=stream)
        return self.y

    def select(self, dy: torch.Tensor, quota: torch.Tensor | None, stream=None) -> None:
        r = self.record
        _lib.moe_select_retained(self.dims, self.ws, dy, quota, self.ret_offsets if r else None,
                                 self.ret_rows if r else None, self.scores if r else None, stream=stream)

    def backward(self, dy: torch.Tensor, x: torch.Tensor, use_retained: bool, stream=None):
        g = self.grads
        _lib.moe_bwd(self.dims, self.ws, dy, x, use_retained, self.dx, g.get("dw_router"), g.get("dw_gate"),
                     g.get("dw_up"), g.get("dw_down"), g.get("dws_gate"), g.get("dws_up"), g.get("dws_down"),
                     stream=stream)
        return self.dx, g

    def step(self, x: torch.Tensor, dy: torch.Tensor, quota: torch.Tensor | None, stream=None):
        """One training step of the layer: forward, optional retention select, backward."""
        self.forward(x, stream)
        if quota is not None:
            self.select(dy, quota, stream)
        return self.backward(dy, x, quota is not None, stream)
