"""GB300-native (sm_103a) forward and backward of one Folding Tensor and Sequence
Parallelism layer.

The computation lives in libtsp.so (C ABI, include/tsp.h); this package holds the
nvcc build step, a ctypes binding with the C names (argument marshalling only) and
TSPLayer, a small owner of the plan, packed weights and workspace.
"""
from __future__ import annotations

import torch

from ._binding import *  # noqa: F401,F403
from ._binding import __all__ as _binding_all
from ._binding import (tsp_layer_fwd, tsp_layer_fwd_host, tsp_pack_weights, tsp_plan,
                       tsp_plan_batched,
                       tsp_device_status, tsp_packed_weight_bytes, tsp_workspace_bytes,
                       tsp_workspace_init, tsp_attention_fwd, tsp_mlp_fwd, TSPError, TSP_OK,
                       tsp_bwd_workspace_bytes, tsp_layer_bwd, tsp_unpack_weight_grads,
                       tsp_saved_bytes, tsp_layer_fwd_train, tsp_layer_bwd_saved)

__all__ = list(_binding_all) + ["TSPLayer"]


class TSPLayer:
    """One TSP layer on one GPU: plan + packed weights + workspace (all owned here).

    weights: dict of bfloat16 CUDA tensors Wq, Wk, Wv, Wo [H, H], W1, W3 [F, H],
    W2 [H, F] (nn.Linear layout). Activations passed to forward() are in the
    sharded [D, S/D, H] layout (see tsp_shard), or [D, batch, S/D, H] for a
    micro-batch of `batch` sequences.
    """

    def __init__(self, D, S, hidden, heads, ffn, weights, device=None, batch=1):
        self.device = torch.device(device or "cuda")
        self.plan = (tsp_plan(D, S, hidden, heads, ffn) if batch == 1
                     else tsp_plan_batched(D, S, batch, hidden, heads, ffn))
        self.wpack = torch.empty(tsp_packed_weight_bytes(self.plan) // 2, dtype=torch.bfloat16,
                                 device=self.device)
        self.ws = torch.empty(tsp_workspace_bytes(self.plan), dtype=torch.uint8, device=self.device)
        tsp_workspace_init(self.plan, self.ws)
        tsp_pack_weights(self.plan, *(weights[k] for k in ("Wq", "Wk", "Wv", "Wo", "W1", "W3", "W2")),
                         self.wpack)

    @property
    def shape(self):
        i = self.plan.info
        return (i.D, i.T, i.hidden) if i.batch == 1 else (i.D, i.batch, i.T, i.hidden)

    def _out(self, out):
        if out is None:
            out = torch.empty(self.shape, dtype=torch.bfloat16, device=self.device)
        return out

    def forward(self, xs, out=None, stream=None):
        out = self._out(out)
        tsp_layer_fwd(self.plan, xs, self.wpack, out, self.ws, stream)
        return out

    def attention(self, xs, out=None, stream=None):
        out = self._out(out)
        tsp_attention_fwd(self.plan, xs, self.wpack, out, self.ws, stream)
        return out

    def mlp(self, hs, out=None, stream=None):
        out = self._out(out)
        tsp_mlp_fwd(self.plan, hs, self.wpack, out, self.ws, stream)
        return out

    def enable_backward(self):
        """Grow the workspace to the backward's size (it serves the forward too)."""
        need = tsp_bwd_workspace_bytes(self.plan)
        if self.ws.numel() < need:
            self.ws = torch.empty(need, dtype=torch.uint8, device=self.device)
            tsp_workspace_init(self.plan, self.ws)

    def backward(self, xs, dout, dxs=None, dwpack=None, stream=None):
        """Gradients of forward(xs) for the output gradient dout (sharded layout):
        returns (dxs, dwpack), dwpack the packed fp32 weight gradients (see
        weight_grads)."""
        self.enable_backward()
        dxs = self._out(dxs)
        if dwpack is None:
            dwpack = torch.empty(self.plan.info.wpack_elems, dtype=torch.float32,
                                 device=self.device)
        tsp_layer_bwd(self.plan, xs, self.wpack, dout, dxs, dwpack, self.ws, stream)
        return dxs, dwpack

    def forward_train(self, xs, out=None, saved=None, stream=None):
        """forward() that also keeps what backward_saved() needs; returns (out, saved)."""
        self.enable_backward()
        out = self._out(out)
        if saved is None:
            saved = torch.empty(tsp_saved_bytes(self.plan), dtype=torch.uint8, device=self.device)
        tsp_layer_fwd_train(self.plan, xs, self.wpack, out, saved, self.ws, stream)
        return out, saved

    def backward_saved(self, xs, saved, dout, dxs=None, dwpack=None, stream=None):
        """backward() from the `saved` of forward_train(xs): same results, without
        running the attention forward again."""
        self.enable_backward()
        dxs = self._out(dxs)
        if dwpack is None:
            dwpack = torch.empty(self.plan.info.wpack_elems, dtype=torch.float32,
                                 device=self.device)
        tsp_layer_bwd_saved(self.plan, xs, self.wpack, saved, dout, dxs, dwpack, self.ws, stream)
        return dxs, dwpack

    def weight_grads(self, dwpack, stream=None):
        """Packed fp32 weight gradients -> dict of nn.Linear-layout fp32 tensors."""
        i = self.plan.info
        H, F = i.hidden, i.ffn
        out = {k: torch.empty(shape, dtype=torch.float32, device=self.device) for k, shape in (
            ("dWq", (H, H)), ("dWk", (H, H)), ("dWv", (H, H)), ("dWo", (H, H)),
            ("dW1", (F, H)), ("dW3", (F, H)), ("dW2", (H, F)))}
        tsp_unpack_weight_grads(self.plan, dwpack, stream=stream, **out)
        return out

    def forward_host(self, x_host, out_host, stream=None):
        tsp_layer_fwd_host(self.plan, x_host, self.wpack, out_host, self.ws, stream)
        return out_host

    def check(self, stream=None):
        """Synchronise and raise TSPError if a bounded device wait gave up."""
        st = tsp_device_status(self.ws, stream)
        if st != TSP_OK:
            from ._binding import tsp_last_error
            raise TSPError(st, tsp_last_error())
